"""Helpers shared by the GPU tests: device upload of seeded inputs, calls
through the C ABI, and the comparison against the FP64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from block_scaled_fp4_moe_gb300 import inputs, moe


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return inputs.bf16_bits_to_f32(bits).astype(np.float64)


class Problem:
    """Host arrays + device copies of one layer instance."""

    def __init__(self, x, wr, bias, bank_np, E, top_k, has_shared=1, shared_weight=1.0):
        self.x, self.wr, self.bias, self.bank_np = x, wr, bias, bank_np
        self.E, self.top_k, self.has_shared, self.shared_weight = E, top_k, has_shared, shared_weight
        self.T, self.H = x.shape
        self.kps = top_k + has_shared
        self.bank = moe.MXFP4Bank.from_host(bank_np, E, has_shared)      # uploads and repacks
        self.xd = dev_bf16(x)
        self.wrd = torch.from_numpy(wr).cuda()
        self.bd = None if bias is None else torch.from_numpy(bias).cuda()

    @staticmethod
    def from_config(cfg: inputs.MoEConfig, bank_np=None) -> "Problem":
        x = inputs.make_x(cfg)
        wr, bias = inputs.make_router(cfg)
        if bank_np is None:
            bank_np = inputs.make_bank(cfg)
        return Problem(x, wr, bias, bank_np, cfg.E, cfg.top_k, cfg.has_shared)

    def expert(self, e):
        return {k: v[e] for k, v in self.bank_np.items()}

    def workspace(self):
        return moe.alloc_workspace(self.T, self.bank, self.top_k)

    def forward(self, ws=None):
        ws = self.workspace() if ws is None else ws
        y = torch.full((self.T, self.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        ids = torch.full((self.T, self.kps), -1, dtype=torch.int32, device="cuda")
        w = torch.full((self.T, self.kps), float("nan"), dtype=torch.float32, device="cuda")
        moe.moe_layer_forward(self.xd, self.wrd, self.bd, self.top_k, self.bank, self.shared_weight, y, ids, w, ws)
        st = moe.moe_check_device_status(ws)
        assert st == 0, moe.moe_status_string(st)
        return {"y": host_bits(y), "ids": ids.cpu().numpy(), "w": w.cpu().numpy(), "ws": ws}

    def grouping(self, ws):
        """The grouping the layer call left in its workspace (a3), in the form
        oracle.group returns."""
        kps, n_tot = self.kps, self.E + self.has_shared
        host = ws.cpu().numpy()

        def region(name, count):
            off = moe.moe_workspace_offset(self.T, self.H, self.bank.inter, self.E, self.top_k, self.has_shared, name)
            return host[off: off + 4 * count].view(np.int32).copy()
        na = int(region("num_active", 1)[0])
        n = self.T * kps
        return {"offsets": region("offsets", n_tot + 1), "sorted_tok": region("sorted_tok", n),
                "sorted_slot": region("sorted_slot", n), "active": region("active", n_tot)[:na],
                "num_active": na, "inv_pos": region("inv_pos", n)}

    def oracle_route(self):
        return oracle.route(self.x, self.wr, self.bias, self.top_k, self.has_shared, self.shared_weight)

    def oracle_tokens(self, route, tokens):
        return oracle.moe_tokens(self.x, route["ids"], route["w"], self.expert, tokens)


def check_grouping(got: dict, ids: np.ndarray, n_tot: int, label: str = "") -> None:
    """Bit-exact grouping against the oracle's, and the inverse permutation."""
    g = oracle.group(ids, n_tot)
    for key in ("offsets", "sorted_tok", "sorted_slot", "active"):
        np.testing.assert_array_equal(got[key], g[key], err_msg=f"{label}: {key}")
    assert got["num_active"] == g["num_active"], label
    kps = ids.shape[1]
    entry = g["sorted_tok"] * kps + g["sorted_slot"]          # sorted position -> entry
    np.testing.assert_array_equal(got["inv_pos"][entry], np.arange(entry.size), err_msg=f"{label}: inv_pos")


def check_output(y_bits: np.ndarray, ref: np.ndarray, label: str = "") -> dict:
    """Tolerance of the layer output: max|err| <= 2e-2 max|ref| and
    mean|err| / mean|ref| <= 5e-3 (the problem statement's bound), plus the
    bound the kernels' arithmetic gives: half a bf16 unit of the reference
    (the final rounding) plus 1e-4 of the token's rms output (fp32
    accumulation, f16 activation splitting)."""
    y = bf16_to_f64(y_bits)
    err = np.abs(y - ref)
    aref = np.abs(ref)
    stats = {"max_err": float(err.max()), "max_ref": float(aref.max()),
             "mean_rel": float(err.mean() / aref.mean()),
             "exact_bf16": float(np.mean(y_bits == oracle.bf16_round_array(ref)))}
    assert np.all(np.isfinite(y)), label
    assert err.max() <= 2e-2 * aref.max(), (label, stats)
    assert err.mean() / aref.mean() <= 5e-3, (label, stats)
    ulp = np.exp2(np.floor(np.log2(np.maximum(aref, 1e-30))) - 7)
    rms = np.sqrt(np.mean(ref ** 2, axis=-1, keepdims=True))
    bound = 0.5 * ulp * (1 + 1e-6) + 1e-4 * rms
    bad = err > bound
    assert not bad.any(), (label, stats, int(bad.sum()), float((err / bound).max()))
    return stats


def random_problem(T, H, E, k, I, has_shared=1, seed=0, bias=True, shared_weight=1.0):
    rng = np.random.default_rng(seed)
    x = inputs.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    wr = (0.02 * rng.standard_normal((H, E))).astype(np.float32)
    b = (0.05 * rng.standard_normal(E)).astype(np.float32) if bias else None
    n = E + has_shared
    bank = {"w13": rng.integers(0, 256, (n, 2 * I, H // 2), dtype=np.uint8),
            "s13": rng.integers(118, 125, (n, 2 * I, H // 32), dtype=np.uint8),
            "w2": rng.integers(0, 256, (n, H, I // 2), dtype=np.uint8),
            "s2": rng.integers(118, 125, (n, H, I // 32), dtype=np.uint8)}
    return Problem(x, wr, b, bank, E, k, has_shared, shared_weight)
