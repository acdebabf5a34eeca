"""GPU parity of the per-(token, group) send runs: the run tables against the
oracle's group_runs, the send buffer (codes and scales) against its
dispatch_runs, both bit-exact, and GEMM1 through the row gather within the
stated tolerance of the oracle's GEMM1 -- and bit-for-bit the dense GEMM1's
output, since every dense row reads the same codes and scales either way."""
import numpy as np
import pytest
import torch

import combine_counting_sort_gb300 as moe
import oracle
from combine_counting_sort_gb300 import inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gu.build()


def runs_of(ids, w, E, G):
    L, st = gu.gpu_layout(ids, w, E, G)
    S = moe.SendRuns(L)
    for t in S.t.values():
        t.fill_(-9)
    moe.moe_send_layout(torch.from_numpy(ids).cuda(), L, S, st)
    torch.cuda.synchronize()
    return L, S, st


def check_tables(S, ref_layout, ids, E, G):
    ref = oracle.group_runs(ids, E, G, ref_layout["row_pair"])
    got = S.numpy()
    n = int(ref["run_offset"][-1])
    assert np.array_equal(got["run_offset"], ref["run_offset"])
    assert np.array_equal(got["send_token"][:n], ref["send_token"])
    assert np.all(got["send_token"][n:] == -1)
    assert np.array_equal(got["send_row"], ref["send_row"].reshape(-1))
    assert np.array_equal(got["run_ready"], ref["run_ready"])
    R = int(ref_layout["expert_offset"][-1])
    assert np.array_equal(got["gather_row"][:R], ref["gather_row"][:R])
    assert np.all(got["gather_row"][R:] == -1)
    return ref


@pytest.mark.parametrize("name", ["tiny", "t2048_uniform", "t8192_zipf1.2", "stage1_t16384_zipf1.0"])
def test_send_runs_tables_match_oracle(name):
    cfg = inputs.CONFIGS[name]
    ids, w = gu.routed(cfg)
    L, S, st = runs_of(ids, w, cfg.E, cfg.G)
    assert st.item() == 0
    check_tables(S, oracle.route_layout(ids, w, cfg.E, cfg.G), ids, cfg.E, cfg.G)


@pytest.mark.parametrize("T,k,E,G", [(1, 1, 4, 2), (37, 4, 16, 1), (300, 4, 16, 16), (129, 8, 64, 32),
                                     (700, 3, 12, 4)])
def test_send_runs_shapes_and_duplicates(T, k, E, G):
    rng = np.random.default_rng(T * 7 + G)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)      # duplicates within a token allowed
    w = rng.random((T, k)).astype(np.float32)
    L, S, st = runs_of(ids, w, E, G)
    assert st.item() == 0
    check_tables(S, oracle.route_layout(ids, w, E, G), ids, E, G)


def dispatch_both(cfg, ids, w, W=None):
    x = inputs.make_x(cfg.T, cfg.H, cfg.seed)
    L, S, st = runs_of(ids, w, cfg.E, cfg.G)
    smax = S.max_rows
    A_send = torch.full((smax, cfg.H), 0xEE, dtype=torch.uint8, device="cuda")
    As_send = torch.full((cfg.H // 128, smax), float("nan"), dtype=torch.float32, device="cuda")
    moe.moe_dispatch_quant_runs(x.cuda(), L, S, A_send, As_send, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return x, L, S, A_send, As_send, st


@pytest.mark.parametrize("name", ["tiny", "t2048_uniform", "t8192_zipf1.2"])
def test_send_buffer_matches_oracle(name):
    cfg = inputs.CONFIGS[name]
    ids, w = gu.routed(cfg)
    x, L, S, A_send, As_send, _ = dispatch_both(cfg, ids, w)
    ref = oracle.group_runs(ids, cfg.E, cfg.G, oracle.route_layout(ids, w, cfg.E, cfg.G)["row_pair"])
    n = int(ref["run_offset"][-1])
    rows = np.arange(n) if n <= 4096 else np.unique(np.random.default_rng(1).choice(n, 2048, replace=False))
    toks = ref["send_token"][rows]
    q, s = oracle.quantize_rows(inputs.bf16_bits(x[torch.as_tensor(toks.astype(np.int64))]))
    Aw, Sw = oracle.dispatch_runs(q, s, np.arange(len(rows)))
    assert np.array_equal(A_send.cpu().numpy()[rows], Aw)
    assert np.array_equal(As_send.cpu().numpy()[:, rows].view(np.uint32), Sw.view(np.uint32))
    # the send buffer holds 1.4-1.6 rows fewer per token than the dense buffer's k
    if cfg.k == 8:
        assert 1.3 < cfg.T * cfg.k / n < 1.7


@pytest.mark.parametrize("T,H,E,G,k,N,skew", [
    (128, 256, 8, 2, 2, 512, None),
    (300, 512, 16, 4, 4, 512, 1.3),
    (700, 1024, 32, 8, 8, 768, 1.2),
    (1, 256, 4, 2, 1, 256, None),
])
def test_gemm1_gather_matches_oracle_and_dense(T, H, E, G, k, N, skew):
    cfg = inputs.MoEConfig("runs", T=T, H=H, E=E, G=G, k=k, N=N, zipf=skew, seed=5)
    ids, w = gu.routed(cfg)
    x, L, S, A_send, As_send, st = dispatch_both(cfg, ids, w)
    W = inputs.make_weights(E, N, H, seed=5).cuda()
    Wq = torch.empty(E, N, H, dtype=torch.uint8, device="cuda")
    Ws = torch.empty(E, N // 128, H // 128, dtype=torch.float32, device="cuda")
    moe.moe_quant_weights(W, Wq, Ws)
    R = T * k
    Yg = torch.full((R + 128, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_gemm1_gather(A_send, As_send, Wq, Ws, L, S, Yg[:R], st)
    A = torch.empty(R, H, dtype=torch.uint8, device="cuda")
    As = torch.empty(H // 128, R, dtype=torch.float32, device="cuda")
    Yd = torch.full((R, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_dispatch_quant(x.cuda(), L, A, As, st)
    moe.moe_grouped_gemm1(A, As, Wq, Ws, L, Yd, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(Yg[:R].view(torch.int16), Yd.view(torch.int16))
    assert torch.isnan(Yg[R:].float()).all()
    # against the oracle, from its own operands
    ref = oracle.route_layout(ids, w, E, G)
    q, s = oracle.quantize_rows(inputs.bf16_bits(x))
    Ad, Asd = oracle.dispatch(q, s, ref["pair_row"], k)
    Wq_ref, Ws_ref = oracle.quantize_weights(inputs.bf16_bits(W))
    want = oracle.grouped_gemm1(Ad, Asd, Wq_ref, Ws_ref, ref["expert_offset"])
    gu.assert_close_bf16(gu.bits(Yg[:R]), want, "gemm1_gather")


def test_gemm1_gather_full_size_matches_dense():
    cfg = inputs.CONFIGS["t8192_zipf1.2"]
    ids, w = gu.routed(cfg)
    x, L, S, A_send, As_send, st = dispatch_both(cfg, ids, w)
    W = inputs.make_weights(cfg.E, cfg.N, cfg.H, cfg.seed, device="cuda")
    Wq = torch.empty(cfg.E, cfg.N, cfg.H, dtype=torch.uint8, device="cuda")
    Ws = torch.empty(cfg.E, cfg.N // 128, cfg.H // 128, dtype=torch.float32, device="cuda")
    moe.moe_quant_weights(W, Wq, Ws)
    del W
    R = cfg.T * cfg.k
    Yg = torch.empty(R, cfg.N, dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_gemm1_gather(A_send, As_send, Wq, Ws, L, S, Yg, st)
    A = torch.empty(R, cfg.H, dtype=torch.uint8, device="cuda")
    As = torch.empty(cfg.H // 128, R, dtype=torch.float32, device="cuda")
    Yd = torch.empty(R, cfg.N, dtype=torch.bfloat16, device="cuda")
    moe.moe_dispatch_quant(x.cuda(), L, A, As, st)
    moe.moe_grouped_gemm1(A, As, Wq, Ws, L, Yd, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(Yg.view(torch.int16), Yd.view(torch.int16))
