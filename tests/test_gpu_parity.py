"""Parity of the CUDA path (through the C ABI) with the FP64 oracle.

Routing and grouping must match exactly; the bf16 layer output must meet
max|err| <= 2e-2 max|ref| and mean|err|/mean|ref| <= 5e-3, and the tighter
bound derived from the kernels' arithmetic (see gpu_support.check_output).
Every shape, small or full size, is compared element by element on every
token; the grouping the call leaves in its workspace is compared with the
oracle's bit for bit.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_moe_gb300 import _build, inputs, moe
from gpu_support import Problem, check_grouping, check_output, dev_bf16, host_bits, random_problem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    moe.lib()
    torch.cuda.init()


def compare_all(p: Problem, label: str):
    out = p.forward()
    r = p.oracle_route()
    np.testing.assert_array_equal(out["ids"], r["ids"], err_msg=label)
    check_grouping(p.grouping(out["ws"]), r["ids"], p.E + p.has_shared, label)
    np.testing.assert_allclose(out["w"], r["w"], rtol=2e-6, atol=1e-7, err_msg=label)
    ref = p.oracle_tokens(r, np.arange(p.T))["y"]
    return check_output(out["y"], ref, label)


# ------------------------------------------------------------- building blocks

def test_e2m1_decode_lane_layout():
    codes = torch.arange(256, dtype=torch.uint8, device="cuda")
    out = torch.empty(512, dtype=torch.int16, device="cuda")
    moe.moe_selftest_decode_e2m1(codes, out)
    got = out.cpu().numpy().view(np.uint16)
    mag = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)
    val = np.concatenate([mag, -mag]).astype(np.float16).view(np.uint16)
    val[8] = 0x8000                                   # -0
    want = np.stack([val[np.arange(256) & 15], val[np.arange(256) >> 4]], axis=1).ravel()
    np.testing.assert_array_equal(got, want)


def numpy_pack_section(codes, scales, row_of):
    """The documented repacked order of one section, written with numpy:
    codes [n, R, K/2], scales [n, R, K/32]; row_of(rb, m) -> canonical row."""
    n, R, Kh = codes.shape
    K = 2 * Kh
    out = []
    for e in range(n):
        for rb in range(row_of.n_rb):
            rows = [row_of(rb, m) for m in range(16)]
            for q in range(K // 64):
                step = np.zeros(544, dtype=np.uint8)
                for lane in range(32):
                    g, c = lane // 4, lane % 4
                    words = []
                    for blk, m in ((2 * q, g), (2 * q, g + 8), (2 * q + 1, g), (2 * q + 1, g + 8)):
                        words.append(codes[e, rows[m], 16 * blk + 4 * c: 16 * blk + 4 * c + 4])
                    step[16 * lane: 16 * lane + 16] = np.concatenate(words)
                for g in range(8):
                    step[512 + 4 * g: 516 + 4 * g] = [scales[e, rows[g], 2 * q], scales[e, rows[g], 2 * q + 1],
                                                      scales[e, rows[g + 8], 2 * q], scales[e, rows[g + 8], 2 * q + 1]]
                out.append(step)
    return np.concatenate(out)


class _Rows:
    def __init__(self, n_rb, fn):
        self.n_rb, self.fn = n_rb, fn

    def __call__(self, rb, m):
        return self.fn(rb, m)


def test_pack_bank_matches_documented_layout():
    rng = np.random.default_rng(4)
    E, S, H, I = 3, 1, 128, 192
    n = E + S
    arrs = {"w13": rng.integers(0, 256, (n, 2 * I, H // 2), dtype=np.uint8),
            "s13": rng.integers(0, 256, (n, 2 * I, H // 32), dtype=np.uint8),
            "w2": rng.integers(0, 256, (n, H, I // 2), dtype=np.uint8),
            "s2": rng.integers(0, 256, (n, H, I // 32), dtype=np.uint8)}
    bank = moe.MXFP4Bank.from_host(arrs, E, S, keep_canonical=True)
    torch.cuda.synchronize()
    got = bank.packed.cpu().numpy()
    gu = numpy_pack_section(arrs["w13"], arrs["s13"], _Rows(I // 8, lambda rb, m: 8 * rb + m if m < 8 else I + 8 * rb + m - 8))
    dn = numpy_pack_section(arrs["w2"], arrs["s2"], _Rows(H // 16, lambda rb, m: 16 * rb + m))
    dn_off = (len(gu) + 255) // 256 * 256
    assert got.size == moe.moe_packed_bank_size(H, I, E, S)
    np.testing.assert_array_equal(got[:len(gu)], gu)
    np.testing.assert_array_equal(got[dn_off:dn_off + len(dn)], dn)
    # a permutation: the multiset of bytes is the canonical one
    canon = np.concatenate([a.ravel() for a in arrs.values()])
    np.testing.assert_array_equal(np.bincount(canon, minlength=256),
                                  np.bincount(np.concatenate([gu, dn]), minlength=256))
    # then one exponent base per weight row in unit-row order: 255 where the
    # row holds the NaN exponent, else max(largest exponent - 28, 0)
    def bases(scales, rows):
        s = scales[:, rows, :].astype(np.int64)
        b = np.maximum(s.max(axis=2) - 28, 0)
        b[(s == 255).any(axis=2)] = 255
        return b.astype(np.uint8).ravel()
    gu_rows = [8 * rb + m if m < 8 else I + 8 * rb + m - 8 for rb in range(I // 8) for m in range(16)]
    gu_off = (dn_off + len(dn) + 255) // 256 * 256
    dn_off2 = (gu_off + n * 2 * I + 255) // 256 * 256
    np.testing.assert_array_equal(got[gu_off:gu_off + n * 2 * I], bases(arrs["s13"], gu_rows))
    np.testing.assert_array_equal(got[dn_off2:dn_off2 + n * H], bases(arrs["s2"], list(range(H))))
    assert (got[gu_off:gu_off + n * 2 * I] == 255).any()        # the NaN marker is exercised


def test_group_tokens_matches_oracle():
    rng = np.random.default_rng(2)
    for T, k, E in [(1, 8, 160), (37, 4, 20), (256, 8, 160), (3, 2, 1024)]:
        ids = np.stack([np.concatenate([rng.permutation(E)[:k], [E]]) for _ in range(T)]).astype(np.int32)
        n_tot = E + 1
        dev = lambda n: torch.full((n,), -7, dtype=torch.int32, device="cuda")
        offs, st, ss, act, na = dev(n_tot + 1), dev(T * (k + 1)), dev(T * (k + 1)), dev(n_tot), dev(1)
        ws = torch.zeros(1 << 12, dtype=torch.uint8, device="cuda")
        moe.moe_group_tokens(torch.from_numpy(ids).cuda(), n_tot, offs, st, ss, act, na, ws)
        assert moe.moe_check_device_status(ws) == 0
        g = oracle.group(ids, n_tot)
        np.testing.assert_array_equal(offs.cpu().numpy(), g["offsets"])
        np.testing.assert_array_equal(st.cpu().numpy(), g["sorted_tok"])
        np.testing.assert_array_equal(ss.cpu().numpy(), g["sorted_slot"])
        assert int(na.item()) == g["num_active"]
        np.testing.assert_array_equal(act.cpu().numpy()[: g["num_active"]], g["active"])


def test_group_tokens_rejects_bad_id_on_device():
    ids = torch.tensor([[0, 3, 9]], dtype=torch.int32, device="cuda")   # 9 >= n_tot
    z = lambda n: torch.zeros(n, dtype=torch.int32, device="cuda")
    ws = torch.zeros(1 << 12, dtype=torch.uint8, device="cuda")
    moe.moe_group_tokens(ids, 9, z(10), z(3), z(3), z(9), z(1), ws)
    assert moe.moe_check_device_status(ws) == moe.MOE_ERR_DEVICE_ASSERT
    assert moe.moe_check_device_status(ws) == 0          # cleared


@pytest.mark.parametrize("name", ["glm_zipf_t256", "1t_t8", "tiny"])
def test_route_topk_matches_oracle(name):
    cfg = inputs.CONFIGS[name]
    x = inputs.make_x(cfg)
    wr, bias = inputs.make_router(cfg)
    ids = torch.empty((cfg.T, cfg.slots), dtype=torch.int32, device="cuda")
    w = torch.empty((cfg.T, cfg.slots), dtype=torch.float32, device="cuda")
    ws = torch.zeros(moe.moe_workspace_size(cfg.T, cfg.H, 64, cfg.E, cfg.top_k, 1), dtype=torch.uint8, device="cuda")
    moe.moe_route_topk(dev_bf16(x), torch.from_numpy(wr).cuda(), None if bias is None else torch.from_numpy(bias).cuda(),
                       cfg.top_k, 1, 1.0, ids, w, ws)
    assert moe.moe_check_device_status(ws) == 0
    r = oracle.route(x, wr, bias, cfg.top_k)
    np.testing.assert_array_equal(ids.cpu().numpy(), r["ids"])
    np.testing.assert_allclose(w.cpu().numpy(), r["w"], rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("T,E,k", [(12, 1024, 31), (9, 5, 5), (10, 70, 20), (11, 33, 8)])
def test_route_topk_group_lists_match_the_oracle(T, E, k):
    """Top k at the extremes of the group-list selection (candidates: each
    group of 32 experts' first k ranks, merged by one warp): 32 groups with
    k + 1 = 32 slots, one group holding fewer experts than 32 with k = E, a
    partial last group, and more k than one group's real experts."""
    rng = np.random.default_rng(100 + E)
    H = 512
    x = inputs.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    wr = (0.02 * rng.standard_normal((H, E))).astype(np.float32)
    bias = (0.05 * rng.standard_normal(E)).astype(np.float32)
    ids = torch.empty((T, k + 1), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k + 1), dtype=torch.float32, device="cuda")
    ws = torch.zeros(moe.moe_workspace_size(T, H, 64, E, k, 1), dtype=torch.uint8, device="cuda")
    moe.moe_route_topk(dev_bf16(x), torch.from_numpy(wr).cuda(), torch.from_numpy(bias).cuda(), k, 1, 1.0, ids, w, ws)
    assert moe.moe_check_device_status(ws) == 0
    r = oracle.route(x, wr, bias, k)
    np.testing.assert_array_equal(ids.cpu().numpy(), r["ids"])
    np.testing.assert_allclose(w.cpu().numpy(), r["w"], rtol=2e-6, atol=1e-7)


# ------------------------------------------------------------- whole layer, small

SMALL = [
    dict(T=1, H=1024, E=16, k=4, I=512),
    dict(T=3, H=1024, E=16, k=4, I=512),
    dict(T=8, H=1024, E=16, k=4, I=512),
    dict(T=13, H=1024, E=16, k=4, I=512),          # more tokens than one pass
    dict(T=40, H=1024, E=6, k=3, I=512),           # experts hold up to 40 tokens
    dict(T=80, H=1024, E=4, k=2, I=512),           # several wide passes per expert (tiled kernels)
    dict(T=33, H=1536, E=12, k=3, I=1024, has_shared=0),   # tiled kernels without a shared expert
    dict(T=9, H=1024, E=16, k=8, I=512),           # first T of the multi-launch path
    dict(T=16, H=1024, E=16, k=8, I=512),          # the speculative-verify block size
    dict(T=16, H=1024, E=40, k=8, I=512, has_shared=0),
    dict(T=5, H=1024, E=16, k=4, I=512, has_shared=0),
    dict(T=9, H=320, E=5, k=5, I=192),             # block-mode scales, k == E
    dict(T=2, H=2048, E=4, k=2, I=2048),
    dict(T=6, H=512, E=1024, k=8, I=256),          # large expert count
    dict(T=4, H=1536, E=12, k=3, I=1024, shared_weight=0.5),
]


@pytest.mark.parametrize("case", SMALL, ids=[str(i) for i in range(len(SMALL))])
def test_layer_small_shapes(case):
    p = random_problem(seed=zlib.crc32(str(case).encode()) % 1000, **case)
    compare_all(p, str(case))


@pytest.mark.parametrize("T", [1, 4, 8, 13])
def test_layer_exact_logit_ties_go_to_the_lower_index(T):
    # duplicated router columns give bit-identical logits: four experts tie
    # for the first slots across both groups of 32, and three more tie at the
    # k-th slot, so the cut falls inside a tie (lower indices win)
    p = random_problem(T=T, H=1024, E=64, k=6, I=512, seed=31 + T, bias=False)
    rng = np.random.default_rng(7)
    base = inputs.bf16_bits_to_f32(p.x[0])
    x = base[None, :] + 0.1 * rng.standard_normal((T, p.H)).astype(np.float32)
    p.x = inputs.f32_to_bf16_bits(x.astype(np.float32))
    p.xd = dev_bf16(p.x)
    v = (0.02 * np.sign(base)).astype(np.float32)
    for e in (3, 17, 35, 50):
        p.wr[:, e] = 3.0 * v
    for e in (8, 40, 41):
        p.wr[:, e] = 1.5 * v
    p.wrd = torch.from_numpy(p.wr).cuda()
    r = p.oracle_route()
    assert (r["ids"][:, :6] == np.array([3, 17, 35, 50, 8, 40])).all()
    compare_all(p, f"ties T={T}")


@pytest.mark.parametrize("T,E,k", [(1, 16, 4), (3, 6, 3), (4, 5, 4), (6, 6, 4), (8, 6, 3), (8, 64, 6), (8, 40, 31)])
def test_layer_grouping_is_the_oracles(T, E, k):
    """The single-launch kernel (T <= 8) groups the entries in shared memory
    on every CTA; CTA 0 leaves that grouping in the workspace.  It must be the
    oracle's bit for bit: few experts make tokens share them (repeated
    experts, groups of several entries), and T * (k + 1) runs from below 32
    entries (the one-warp grouping) to above 32 (the multi-warp one)."""
    p = random_problem(T=T, H=1024, E=E, k=k, I=512, seed=60 + T + E)
    assert moe.moe_layer_launches(T, p.bank, k) == 1
    out = p.forward()
    r = p.oracle_route()
    np.testing.assert_array_equal(out["ids"], r["ids"])
    got = p.grouping(out["ws"])
    check_grouping(got, r["ids"], E + 1, f"T={T} E={E} k={k}")
    if T > 1:
        assert got["num_active"] < T * (k + 1)          # some expert holds several entries
    check_output(out["y"], p.oracle_tokens(r, np.arange(T))["y"], f"grouping case T={T}")


def test_layer_tiny_workload_against_fixture():
    cfg = inputs.CONFIGS["tiny"]
    p = Problem.from_config(cfg)
    stats = compare_all(p, "tiny")
    assert stats["exact_bf16"] >= 0.99


def test_layer_is_deterministic_and_entry_points_agree():
    p = random_problem(T=13, H=1024, E=16, k=4, I=512, seed=5)
    a, b = p.forward(), p.forward()
    np.testing.assert_array_equal(a["y"], b["y"])
    # expert FFN on the layer's own routing gives the same bits
    y2 = torch.empty((p.T, p.H), dtype=torch.bfloat16, device="cuda")
    ws = p.workspace()
    moe.moe_expert_ffn_mxfp4(p.xd, torch.from_numpy(a["ids"]).cuda(), torch.from_numpy(a["w"]).cuda(), p.top_k,
                             p.bank, y2, ws)
    assert moe.moe_check_device_status(ws) == 0
    np.testing.assert_array_equal(host_bits(y2), a["y"])
    # host-memory entry point gives the same bits
    xh = torch.from_numpy(p.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    yh = torch.empty((p.T, p.H), dtype=torch.bfloat16).pin_memory()
    moe.moe_layer_forward_hostio(xh, p.wrd, p.bd, p.top_k, p.bank, 1.0, yh, ws)
    np.testing.assert_array_equal(yh.view(torch.int16).numpy().view(np.uint16), a["y"])


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 6, 7, 8])
def test_single_launch_stages_against_the_oracle(T):
    """The single-launch kernel's intermediate results, entry by entry: h =
    silu(gate) * up (fp32) and each entry's down projection, against the
    oracle's, three calls in a row.  At H = 2048 a row block's steps are split
    across warps, whose partial sums meet in shared memory between the
    shared expert's gate/up units, the routed ones and the down units."""
    p = random_problem(T=T, H=2048, E=24, k=4, I=1024, seed=80 + T)
    assert moe.moe_layer_launches(T, p.bank, p.top_k) == 1
    r = p.oracle_route()
    ref = oracle.moe_tokens(p.x, r["ids"], r["w"], p.expert, np.arange(T), want_h=True, want_slots=True)
    g = oracle.group(r["ids"], p.E + 1)
    n, I, H = T * p.kps, p.bank.inter, p.H
    ws = p.workspace()
    for call in range(3):
        out = p.forward(ws)
        np.testing.assert_array_equal(out["ids"], r["ids"])
        host = ws.cpu().numpy()

        def region(name, cols):
            off = moe.moe_workspace_offset(T, H, I, p.E, p.top_k, 1, name)
            return host[off: off + 4 * n * cols].view(np.float32).reshape(n, cols).astype(np.float64)
        h, ye = region("h", I), region("y_entries", H)
        for pos in range(n):
            t, sl = g["sorted_tok"][pos], g["sorted_slot"][pos]
            hr, yr = ref["h"][t, sl], ref["y_slots"][t, sl]
            assert np.abs(h[pos] - hr).max() <= 1e-5 * np.abs(hr).max(), (call, pos, t, sl)
            assert np.abs(ye[pos] - yr).max() <= 1e-5 * np.abs(yr).max(), (call, pos, t, sl)
        check_output(out["y"], ref["y"], f"stages T={T} call {call}")


@pytest.mark.parametrize("T,H,E,k,I", [(6, 512, 1024, 8, 256), (8, 1024, 160, 8, 512), (1, 1024, 16, 4, 512)])
def test_single_launch_calls_in_a_row_on_one_workspace(T, H, E, k, I):
    """Calls on one workspace leave its counters and router tickets ready for
    the next: five calls in a row give the oracle's routing and bit-identical
    outputs (E = 1024 and T = 8 take the ticketed router sums)."""
    p = random_problem(T=T, H=H, E=E, k=k, I=I, seed=70 + T)
    assert moe.moe_layer_launches(T, p.bank, k) == 1
    ws = p.workspace()
    first = p.forward(ws)
    r = p.oracle_route()
    np.testing.assert_array_equal(first["ids"], r["ids"])
    check_output(first["y"], p.oracle_tokens(r, np.arange(T))["y"], f"repeat T={T} E={E}")
    for _ in range(4):
        again = p.forward(ws)
        np.testing.assert_array_equal(again["ids"], first["ids"])
        np.testing.assert_array_equal(again["y"], first["y"])


@pytest.mark.parametrize("T", [1, 4, 13])
def test_chained_layer_hint_changes_nothing(T):
    """moe_layer_forward_next against the oracle, and bit-identical to the
    unchained call (the hint only moves the next layer's bytes into L2)."""
    p = random_problem(T=T, H=1024, E=16, k=4, I=512, seed=40 + T)
    q = random_problem(T=T, H=1024, E=16, k=4, I=512, seed=90 + T)    # the layer that runs next
    a = p.forward()
    r = p.oracle_route()
    ref = p.oracle_tokens(r, np.arange(T))["y"]
    for nr, nb in ((q.wrd, q.bank), (None, q.bank), (q.wrd, None), (None, None)):
        ws = p.workspace()
        y = torch.full((p.T, p.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        ids = torch.full((p.T, p.kps), -1, dtype=torch.int32, device="cuda")
        w = torch.full((p.T, p.kps), float("nan"), dtype=torch.float32, device="cuda")
        moe.moe_layer_forward_next(p.xd, p.wrd, p.bd, p.top_k, p.bank, p.shared_weight, y, ids, w, ws,
                                   next_router_w=nr, next_bank=nb)
        assert moe.moe_check_device_status(ws) == 0
        np.testing.assert_array_equal(ids.cpu().numpy(), r["ids"])
        check_output(host_bits(y), ref, f"chained T={T}")
        np.testing.assert_array_equal(host_bits(y), a["y"])
        np.testing.assert_array_equal(ids.cpu().numpy(), a["ids"])
        np.testing.assert_array_equal(w.cpu().numpy(), a["w"])


def test_zero_tokens_is_a_noop():
    p = random_problem(T=1, H=1024, E=16, k=4, I=512)
    y = torch.empty((0, p.H), dtype=torch.bfloat16, device="cuda")
    x = torch.empty((0, p.H), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(moe.moe_workspace_size(0, p.H, 512, 16, 4, 1) + 256, dtype=torch.uint8, device="cuda")
    moe.moe_layer_forward(x, p.wrd, p.bd, 4, p.bank, 1.0, y, ws=ws)
    torch.cuda.synchronize()


def test_bad_routing_is_reported_and_leaves_outputs_untouched():
    """A caller-supplied expert id out of range is caught on the device: the
    status word reports it, y keeps its contents, and the next call works."""
    p = random_problem(T=3, H=1024, E=16, k=4, I=512, seed=9)
    ws = p.workspace()
    ids = torch.tensor([[0, 1, 2, 3, 16], [4, 5, 6, 99, 16], [1, 2, 3, 4, 16]], dtype=torch.int32, device="cuda")
    w = torch.full((3, 5), 0.25, dtype=torch.float32, device="cuda")
    y = torch.full((p.T, p.H), 7.0, dtype=torch.bfloat16, device="cuda")
    moe.moe_expert_ffn_mxfp4(p.xd, ids, w, p.top_k, p.bank, y, ws)
    assert moe.moe_check_device_status(ws) == moe.MOE_ERR_DEVICE_ASSERT
    assert torch.all(y == 7.0)
    out = p.forward(ws)                                    # the context is still usable
    r = p.oracle_route()
    check_output(out["y"], p.oracle_tokens(r, np.arange(p.T))["y"], "after a rejected call")


# ------------------------------------------------------ full-size workloads

# every token of every full-size workload is compared with the oracle
FULL = ["glm_t1", "glm_verify_t4", "glm_verify_t16", "glm_zipf_t64", "glm_zipf_t256", "1t_t1", "1t_t4", "1t_t8"]


@pytest.fixture(scope="module")
def banks():
    cache = {}

    def get(cfg):
        key = (cfg.H, cfg.E, cfg.I, cfg.seed)
        if key not in cache:
            cache.clear()
            torch.cuda.empty_cache()
            cache[key] = inputs.make_bank(cfg)
        return cache[key]
    return get


@pytest.mark.parametrize("name", FULL)
def test_layer_full_size(name, banks):
    """Full-size workloads in the launch form the benchmark times: routing
    and grouping bit-exact, every token's output within the tolerance."""
    cfg = inputs.CONFIGS[name]
    p = Problem.from_config(cfg, banks(cfg))
    out = p.forward()
    r = p.oracle_route()
    np.testing.assert_array_equal(out["ids"], r["ids"])
    np.testing.assert_allclose(out["w"], r["w"], rtol=2e-6, atol=1e-7)
    check_grouping(p.grouping(out["ws"]), r["ids"], cfg.E + cfg.has_shared, name)
    ref = p.oracle_tokens(r, np.arange(cfg.T, dtype=np.int32))["y"]
    check_output(out["y"], ref, name)
    del p
    torch.cuda.empty_cache()


# ------------------------------------------------- single-launch kernel


def test_device_wait_limit_reports_timeout_and_workspace_stays_usable():
    """A grid wait that nothing completes gives up after its limit; the
    status word says so and the same workspace then runs a correct layer."""
    p = random_problem(T=2, H=1024, E=16, k=4, I=512, seed=21)
    ws = p.workspace()
    moe.moe_selftest_wait_timeout(ws)
    assert moe.moe_check_device_status(ws) == moe.MOE_ERR_DEVICE_TIMEOUT
    out = p.forward(ws)
    r = p.oracle_route()
    np.testing.assert_array_equal(out["ids"], r["ids"])
    check_output(out["y"], p.oracle_tokens(r, np.arange(p.T))["y"], "after a timed-out wait")


def test_launch_count_and_phase_times():
    p = random_problem(T=1, H=1024, E=16, k=4, I=512, seed=22)
    assert moe.moe_layer_launches(1, p.bank, p.top_k) == 1
    assert moe.moe_layer_launches(8, p.bank, p.top_k) == 1
    assert moe.moe_layer_launches(9, p.bank, p.top_k) == 6
    assert moe.moe_layer_launches(16, p.bank, p.top_k) == 6
    assert moe.moe_layer_launches(0, p.bank, p.top_k) == 0
    out = p.forward()
    ph = moe.moe_read_phase_times(out["ws"])
    assert all(v >= 0.0 for v in ph.values()), ph
    assert 0.0 < ph["total"] < 1e5, ph
