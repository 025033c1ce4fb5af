"""The allocation-free entry point, moe_layer_forward_noalloc.

Some callers cannot allocate device memory themselves (plugins whose host
application owns every device allocation, runtimes with a device-memory
budget fixed at start-up).  For them the library runs the layer on a scratch
array compiled into it.  This test calls that entry point through the C ABI
twice in a row and checks each result against the workspace entry point
moe_layer_forward: both run the same kernels on the same inputs, so y, the
expert ids and the weights must agree bit for bit (which is within every
tolerance the other parity tests use).  It sits
in a file of its own that pytest collects last, and passes both alone in a
fresh process (where its first call does the per-device set-up) and after the
other tests.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from block_scaled_fp4_moe_gb300 import _build, inputs, moe
from gpu_support import Problem, host_bits

pytestmark = pytest.mark.gpu


def _problem(T, H, E, k, I, seed):
    rng = np.random.default_rng(seed)
    x = inputs.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    wr = (0.02 * rng.standard_normal((H, E))).astype(np.float32)
    b = (0.05 * rng.standard_normal(E)).astype(np.float32)
    n = E + 1
    bank = {"w13": rng.integers(0, 256, (n, 2 * I, H // 2), dtype=np.uint8),
            "s13": rng.integers(118, 125, (n, 2 * I, H // 32), dtype=np.uint8),
            "w2": rng.integers(0, 256, (n, H, I // 2), dtype=np.uint8),
            "s2": rng.integers(118, 125, (n, H, I // 32), dtype=np.uint8)}
    return Problem(x, wr, b, bank, E, k)


@pytest.mark.parametrize("shape", [dict(T=1, H=1024, E=16, k=4, I=512), dict(T=5, H=2048, E=24, k=6, I=1024)])
def test_noalloc_matches_workspace_entry_point_twice(shape):
    _build.build()
    p = _problem(seed=11, **shape)
    ref = p.forward()                                      # moe_layer_forward with its own workspace
    b = p.bank.c_struct()
    for call in range(2):
        y = torch.full((p.T, p.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        ids = torch.full((p.T, p.kps), -1, dtype=torch.int32, device="cuda")
        w = torch.full((p.T, p.kps), float("nan"), dtype=torch.float32, device="cuda")
        st = moe.lib().moe_layer_forward_noalloc(
            C.c_void_p(p.xd.data_ptr()), C.c_void_p(p.wrd.data_ptr()), C.c_void_p(p.bd.data_ptr()), p.T, p.top_k,
            C.byref(b), 1.0, C.c_void_p(y.data_ptr()), C.c_void_p(ids.data_ptr()), C.c_void_p(w.data_ptr()),
            C.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == moe.MOE_OK, moe.moe_status_string(st)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(ids.cpu().numpy(), ref["ids"], err_msg=f"call {call}")
        np.testing.assert_array_equal(w.cpu().numpy(), ref["w"], err_msg=f"call {call}")
        np.testing.assert_array_equal(host_bits(y), ref["y"], err_msg=f"noalloc call {call}")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    _build.build()
    p = _problem(T=1, H=1024, E=16, k=4, I=512, seed=3)
    b = p.bank.c_struct()
    T = 4096                                                 # workspace far above the built-in array
    assert moe.moe_workspace_size(T, p.H, 512, 16, 4, 1) > 16 << 20
    st = moe.lib().moe_layer_forward_noalloc(
        C.c_void_p(p.xd.data_ptr()), C.c_void_p(p.wrd.data_ptr()), None, T, p.top_k, C.byref(b), 1.0,
        C.c_void_p(p.xd.data_ptr()), None, None, C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == moe.MOE_ERR_WORKSPACE_TOO_SMALL
