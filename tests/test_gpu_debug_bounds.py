"""The range-checking build (libmoe_fp4_debug.so, compiled with
MOE_DEBUG_BOUNDS): every access whose index comes from routing data --
sorted positions, window rows, output rows -- is checked on the device, and a
failed check reports MOE_ERR_DEVICE_ASSERT instead of touching memory.

Each launch form runs under that build (the single-launch kernel at T <= 8,
the multi-launch kernels above, the expert FFN on caller routing, the MXFP8
variant); no check may fire, the routing must be the oracle's and the
outputs within the parity tests' tolerance of it.  (The two builds are
different binaries, so the compiler may contract multiply-adds differently:
the outputs may differ from the normal build's in the last bit, but repeated
calls of the debug build agree bit for bit.)
"""
import numpy as np
import pytest
import torch

from block_scaled_fp4_moe_gb300 import _build, inputs, moe
from gpu_support import check_output, host_bits, random_problem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    _build.build(debug=True)
    torch.cuda.init()


def run_layer(p, mx=False):
    ws = p.workspace()
    y = torch.full((p.T, p.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    ids = torch.full((p.T, p.kps), -1, dtype=torch.int32, device="cuda")
    w = torch.full((p.T, p.kps), float("nan"), dtype=torch.float32, device="cuda")
    layer = moe.moe_layer_forward_mxfp8 if mx else moe.moe_layer_forward
    layer(p.xd, p.wrd, p.bd, p.top_k, p.bank, p.shared_weight, y, ids, w, ws)
    st = moe.moe_check_device_status(ws)
    return st, host_bits(y), ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("T,H,E,k,I", [(1, 1024, 16, 4, 512), (5, 1024, 16, 4, 512), (8, 2048, 24, 4, 1024),
                                        (6, 512, 1024, 8, 256), (13, 1024, 16, 4, 512), (40, 1024, 6, 3, 512),
                                        (80, 1024, 4, 2, 512), (9, 320, 5, 5, 192)])
def test_debug_build_fires_no_check_and_matches(T, H, E, k, I):
    p = random_problem(T=T, H=H, E=E, k=k, I=I, seed=100 + T)
    st0, y0, ids0, w0 = run_layer(p)
    assert st0 == 0
    with moe.debug_bounds():
        st1, y1, ids1, w1 = run_layer(p)
        assert st1 == 0, moe.moe_status_string(st1)
        # the expert FFN on the layer's own routing
        ws = p.workspace()
        y2 = torch.empty((p.T, p.H), dtype=torch.bfloat16, device="cuda")
        moe.moe_expert_ffn_mxfp4(p.xd, torch.from_numpy(ids0).cuda(), torch.from_numpy(w0).cuda(), p.top_k, p.bank,
                                 y2, ws)
        assert moe.moe_check_device_status(ws) == 0
    r = p.oracle_route()
    ref = p.oracle_tokens(r, np.arange(T))["y"]
    np.testing.assert_array_equal(ids1, r["ids"])
    np.testing.assert_allclose(w1, r["w"], rtol=2e-6, atol=1e-7)
    check_output(y1, ref, f"debug build T={T}")
    check_output(host_bits(y2), ref, f"debug build expert FFN T={T}")
    with moe.debug_bounds():
        st3, y3, _, _ = run_layer(p)
    assert st3 == 0
    np.testing.assert_array_equal(y3, y1)


@pytest.mark.parametrize("T", [1, 9])
def test_debug_build_mxfp8_variant(T):
    p = random_problem(T=T, H=1024, E=16, k=4, I=512, seed=120 + T)
    arrays = {key: torch.from_numpy(v).cuda() for key, v in p.bank_np.items()}
    for key, v in arrays.items():
        setattr(p.bank, key, v)
    p.bank.pack_mx()
    st0, y0, ids0, _ = run_layer(p, mx=True)
    assert st0 == 0
    with moe.debug_bounds():
        st1, y1, ids1, _ = run_layer(p, mx=True)
    assert st1 == 0, moe.moe_status_string(st1)
    np.testing.assert_array_equal(ids1, ids0)
    d = np.abs(inputs.bf16_bits_to_f32(y1).astype(np.float64) - inputs.bf16_bits_to_f32(y0))
    assert d.max() <= 1e-2 * np.abs(inputs.bf16_bits_to_f32(y0)).max()


def test_debug_build_split_items():
    """The tensor-memory kernels' leftover items cut along K (tail slots,
    arrival counters, the sum by the last piece's CTA) under the range
    checks: a T = 16 shape with one pass more than fill the SMs at 16 tiles
    per pass and 8 raw stages per item."""
    G = torch.cuda.get_device_properties(0).multi_processor_count
    E = G // 16                              # passes = E + 1 (shared): n_items = 16 (G // 16 + 1) > G
    p = random_problem(T=16, H=4096, E=E, k=min(4, E), I=1024, seed=140)
    with moe.debug_bounds():
        st, y, ids, w = run_layer(p)
    assert st == 0, moe.moe_status_string(st)
    r = p.oracle_route()
    np.testing.assert_array_equal(ids, r["ids"])
    check_output(y, p.oracle_tokens(r, np.arange(p.T))["y"], "debug build split items")
