"""Guard bands around every buffer a call touches (a substitute for a memory
checker, which this machine does not offer).

Each device buffer -- outputs, inputs and the workspace -- is allocated with
4 KB of a known byte pattern before and after it; the workspace is exactly
moe_workspace_size bytes.  Every entry point runs at several sizes (T = 0, 1,
8 -- the single-launch kernel's largest -- 9 and 33, the multi-launch path),
then the test checks that no guard byte changed, that the inputs are
unchanged, and that the outputs are those of an unguarded call.  An
out-of-bounds write within 4 KB of any buffer, or a write to an input, fails.
"""
import numpy as np
import pytest
import torch

from block_scaled_fp4_moe_gb300 import _build, inputs, moe
from gpu_support import Problem, host_bits

pytestmark = pytest.mark.gpu

GUARD = 4096


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    moe.lib()
    torch.cuda.init()


class Guarded:
    """A device tensor with guard bands of a fixed byte pattern on both sides."""

    def __init__(self, nbytes, dtype=torch.uint8, shape=None, fill=None):
        self.nbytes = int(nbytes)
        self.buf = torch.empty(2 * GUARD + self.nbytes, dtype=torch.uint8, device="cuda")
        pat = ((torch.arange(GUARD, device="cuda") * 37 + 11) % 256).to(torch.uint8)
        self.pat = pat
        self.buf[:GUARD] = pat
        self.buf[GUARD + self.nbytes:] = pat
        raw = self.buf[GUARD:GUARD + self.nbytes]
        self.t = raw.view(dtype) if dtype != torch.uint8 else raw
        if shape is not None:
            self.t = self.t.view(shape)
        if fill is not None:
            raw.copy_(fill.contiguous().view(torch.uint8).view(-1))

    def guards_intact(self):
        return bool(torch.equal(self.buf[:GUARD], self.pat) and torch.equal(self.buf[GUARD + self.nbytes:], self.pat))


def guarded_like(t: torch.Tensor) -> Guarded:
    return Guarded(t.numel() * t.element_size(), t.dtype, t.shape, fill=t)


def problem(T, seed=3):
    rng = np.random.default_rng(seed)
    H, E, k, I = 1024, 16, 4, 512
    x = inputs.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    wr = (0.02 * rng.standard_normal((H, E))).astype(np.float32)
    b = (0.05 * rng.standard_normal(E)).astype(np.float32)
    n = E + 1
    bank = {"w13": rng.integers(0, 256, (n, 2 * I, H // 2), dtype=np.uint8),
            "s13": rng.integers(118, 125, (n, 2 * I, H // 32), dtype=np.uint8),
            "w2": rng.integers(0, 256, (n, H, I // 2), dtype=np.uint8),
            "s2": rng.integers(118, 125, (n, H, I // 32), dtype=np.uint8)}
    return Problem(x, wr, b, bank, E, k)


def guarded_ws(T, p):
    n = moe.moe_workspace_size(T, p.H, p.bank.inter, p.E, p.top_k, 1)
    g = Guarded(max(n, 256))
    moe.moe_workspace_init(g.t)
    return g


def inputs_of(p):
    return {"x": guarded_like(p.xd), "wr": guarded_like(p.wrd), "b": guarded_like(p.bd),
            "bank_packed": guarded_like(p.bank.packed)}


def guarded_bank(p, packed):
    return moe.MXFP4Bank(p.E, 1, p.H, p.bank.inter, packed=packed)


def assert_intact(label, bufs, originals=None):
    torch.cuda.synchronize()
    for name, g in bufs.items():
        assert g.guards_intact(), f"{label}: guard band of {name} was written"
    for name, (g, ref) in (originals or {}).items():
        assert torch.equal(g.t.contiguous().view(torch.uint8), ref.contiguous().view(torch.uint8)), \
            f"{label}: input {name} was written"


@pytest.mark.parametrize("T", [0, 1, 8, 9, 33])
def test_layer_forward_stays_inside_its_buffers(T):
    p = problem(max(T, 1))
    if T == 0:
        p.xd = p.xd[:0]
    inp = inputs_of(p)
    bank = guarded_bank(p, inp["bank_packed"].t)
    y = Guarded(T * p.H * 2, torch.bfloat16, (T, p.H))
    ids = Guarded(T * p.kps * 4, torch.int32, (T, p.kps))
    w = Guarded(T * p.kps * 4, torch.float32, (T, p.kps))
    ws = guarded_ws(T, p)
    moe.moe_layer_forward(inp["x"].t, inp["wr"].t, inp["b"].t, p.top_k, bank, 1.0, y.t, ids.t, w.t, ws.t)
    assert moe.moe_check_device_status(ws.t) == 0
    assert_intact(f"moe_layer_forward T={T}", {"y": y, "ids": ids, "w": w, "ws": ws, **inp},
                  {"x": (inp["x"], p.xd), "wr": (inp["wr"], p.wrd), "b": (inp["b"], p.bd),
                   "packed": (inp["bank_packed"], p.bank.packed)})
    if T:
        ref = p.forward()
        np.testing.assert_array_equal(host_bits(y.t), ref["y"])
        np.testing.assert_array_equal(ids.t.cpu().numpy(), ref["ids"])


@pytest.mark.parametrize("T", [1, 9, 33])
def test_route_group_and_expert_ffn_stay_inside_their_buffers(T):
    p = problem(T, seed=5)
    inp = inputs_of(p)
    bank = guarded_bank(p, inp["bank_packed"].t)
    ids = Guarded(T * p.kps * 4, torch.int32, (T, p.kps))
    w = Guarded(T * p.kps * 4, torch.float32, (T, p.kps))
    ws = guarded_ws(T, p)
    moe.moe_route_topk(inp["x"].t, inp["wr"].t, inp["b"].t, p.top_k, 1, 1.0, ids.t, w.t, ws.t)
    assert moe.moe_check_device_status(ws.t) == 0
    n_tot, n = p.E + 1, T * p.kps
    offs, st, ss = Guarded((n_tot + 1) * 4, torch.int32), Guarded(n * 4, torch.int32), Guarded(n * 4, torch.int32)
    act, na = Guarded(n_tot * 4, torch.int32), Guarded(4, torch.int32)
    moe.moe_group_tokens(ids.t, n_tot, offs.t, st.t, ss.t, act.t, na.t, ws.t)
    assert moe.moe_check_device_status(ws.t) == 0
    y = Guarded(T * p.H * 2, torch.bfloat16, (T, p.H))
    moe.moe_expert_ffn_mxfp4(inp["x"].t, ids.t, w.t, p.top_k, bank, y.t, ws.t)
    assert moe.moe_check_device_status(ws.t) == 0
    assert_intact(f"route/group/ffn T={T}",
                  {"ids": ids, "w": w, "ws": ws, "offsets": offs, "sorted_tok": st, "sorted_slot": ss,
                   "active": act, "num_active": na, "y": y, **inp},
                  {"x": (inp["x"], p.xd), "wr": (inp["wr"], p.wrd), "packed": (inp["bank_packed"], p.bank.packed)})
    ref = p.forward()
    np.testing.assert_array_equal(ids.t.cpu().numpy(), ref["ids"])
    assert int(na.t.item()) == len(set(ref["ids"].ravel().tolist()))


@pytest.mark.parametrize("T", [1, 9])
def test_mxfp8_and_chained_entry_points_stay_inside_their_buffers(T):
    p = problem(T, seed=7)
    q = problem(T, seed=8)                                  # the layer named as the next one
    arrays = {k: torch.from_numpy(v).cuda() for k, v in p.bank_np.items()}
    garr = {k: guarded_like(v) for k, v in arrays.items()}
    cbank = moe.MXFP4Bank(p.E, 1, p.H, p.bank.inter, **{k: g.t for k, g in garr.items()})
    packed = Guarded(moe.moe_packed_bank_size(p.H, p.bank.inter, p.E, 1))
    mxn = int(moe.lib().moe_packed_mx_bank_size(p.H, p.bank.inter, p.E, 1))
    packed_mx = Guarded(mxn)
    cbank.packed, cbank.packed_mx = packed.t, packed_mx.t
    cbank.pack()
    cbank.pack_mx()
    inp = inputs_of(p)
    y = Guarded(T * p.H * 2, torch.bfloat16, (T, p.H))
    ws = guarded_ws(T, p)
    moe.moe_layer_forward_mxfp8(inp["x"].t, inp["wr"].t, inp["b"].t, p.top_k, cbank, 1.0, y.t, ws=ws.t)
    assert moe.moe_check_device_status(ws.t) == 0
    y2 = Guarded(T * p.H * 2, torch.bfloat16, (T, p.H))
    qr = guarded_like(q.wrd)
    moe.moe_layer_forward_next(inp["x"].t, inp["wr"].t, inp["b"].t, p.top_k, cbank, 1.0, y2.t, ws=ws.t,
                               next_router_w=qr.t, next_bank=q.bank)
    assert moe.moe_check_device_status(ws.t) == 0
    assert_intact(f"mxfp8/next T={T}",
                  {"y": y, "y2": y2, "ws": ws, "packed": packed, "packed_mx": packed_mx, "next_router": qr,
                   **inp, **{f"bank.{k}": g for k, g in garr.items()}},
                  {"next_router": (qr, q.wrd), **{f"bank.{k}": (g, arrays[k]) for k, g in garr.items()}})
    torch.cuda.synchronize()
    np.testing.assert_array_equal(packed.t.cpu().numpy(), p.bank.packed.cpu().numpy())
    np.testing.assert_array_equal(host_bits(y2.t), p.forward()["y"])
