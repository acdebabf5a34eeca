"""GPU parity of the no-plan small-batch layout (moe_route_layout_noplan)
against the oracle's counting sort.

The no-plan layout places the rows of an expert in reservation order, so
parity is by multiset: every order-free table (counts, offsets, tile tables,
rowmap, group offsets, ready_tokens) must equal the oracle's bit for bit; per
expert the set of pairs held by its rows, and per first expert the set of
tokens in its token-order range, must equal the oracle's; pair_row and
row_pair must be inverse permutations and row_weight must follow row_pair.
Downstream, dispatch -> GEMM1 -> combine through the no-plan layout must give
the counting-sort path's combined output bit for bit (each output row depends
only on its token, expert and weight, not on where the layout put it)."""
import numpy as np
import pytest
import torch

import combine_counting_sort_gb300 as moe
import oracle
from combine_counting_sort_gb300 import inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

ORDER_FREE = ["count", "expert_offset", "expert_tile_offset", "group_offset", "ready_tokens", "rowmap",
              "tile_expert", "tile_row_begin", "tile_rows", "num_tiles"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gu.build()


def noplan_layout(ids, w, E, G, poison=True):
    T, k = ids.shape
    L = moe.Layout(T, k, E, G)
    if poison:
        for t in L.t.values():
            t.fill_(-5)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_route_layout_noplan(torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), L, st)
    torch.cuda.synchronize()
    return L, st


def check_multiset(got: dict, ref: dict, ids: np.ndarray, w: np.ndarray, valid=None):
    T, k = ids.shape
    for name in ORDER_FREE:
        assert np.array_equal(got[name], np.asarray(ref[name])), name
    eo = np.asarray(ref["expert_offset"])
    R = int(eo[-1])
    rp, pr = got["row_pair"][:R], got["pair_row"]
    valid = np.ones(T * k, bool) if valid is None else valid
    assert np.array_equal(rp[pr[valid]], np.nonzero(valid)[0])            # inverse permutations
    assert np.all(pr[~valid] == -1)
    assert np.array_equal(got["row_weight"][:R].view(np.uint32),
                          np.asarray(w, np.float32).reshape(-1)[rp].view(np.uint32))
    for e in range(len(eo) - 1):
        a, b = eo[e], eo[e + 1]
        assert np.array_equal(np.sort(rp[a:b]), np.asarray(ref["row_pair"][a:b])), f"pairs of expert {e}"
    ready = np.asarray(ref["ready_tokens"])
    starts = np.concatenate([[0], ready[:-1]])
    for e in range(len(ready)):
        a, b = starts[e], ready[e]
        assert np.array_equal(np.sort(got["token_order"][a:b]), np.asarray(ref["token_order"][a:b])), \
            f"tokens of first expert {e}"


@pytest.mark.parametrize("T", [8, 32, 128, 256, 1024, 2048])
@pytest.mark.parametrize("zipf", [None, 1.2])
def test_noplan_small_batches(T, zipf):
    cfg = inputs.MoEConfig("np", T=T, H=7168, E=256, G=8, k=8, N=4096, zipf=zipf, seed=T)
    ids, w = gu.routed(cfg)
    L, st = noplan_layout(ids, w, cfg.E, cfg.G)
    assert st.item() == 0
    check_multiset(L.numpy(), oracle.route_layout(ids, w, cfg.E, cfg.G), ids, w)


@pytest.mark.parametrize("T,k,E,G", [(1, 1, 4, 2), (16384, 1, 1024, 4), (2048, 8, 1024, 8), (300, 4, 16, 1),
                                     (5, 32, 32, 4)])
def test_noplan_shapes_and_duplicates(T, k, E, G):
    rng = np.random.default_rng(T + k + E)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)      # duplicates within a token allowed
    if T > 10:
        ids[: T // 3, 0] = 1                                    # skew: one expert holds a third of the batch
    w = rng.random((T, k)).astype(np.float32)
    L, st = noplan_layout(ids, w, E, G)
    assert st.item() == 0
    check_multiset(L.numpy(), oracle.route_layout(ids, w, E, G), ids, w)


def test_noplan_invalid_ids_are_skipped_and_reported():
    rng = np.random.default_rng(9)
    T, k, E, G = 200, 4, 16, 4
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    ids[3, 1], ids[77, 0], ids[150, 3] = -1, E, 1000
    w = rng.random((T, k)).astype(np.float32)
    L, st = noplan_layout(ids, w, E, G)
    assert st.item() == moe.MOE_ERR_EXPERT_ID
    valid = ((ids >= 0) & (ids < E)).reshape(-1)
    # the valid pairs only: counts, offsets, and every row of expert e holding a pair routed to e
    got = L.numpy()
    counts = np.bincount(ids.reshape(-1)[valid], minlength=E)
    assert np.array_equal(got["count"], counts)
    eo = np.concatenate([[0], np.cumsum(counts)])
    assert np.array_equal(got["expert_offset"], eo)
    rp, pr = got["row_pair"][: eo[-1]], got["pair_row"]
    assert np.array_equal(rp[pr[valid]], np.nonzero(valid)[0]) and np.all(pr[~valid] == -1)
    for e in range(E):
        held = ids.reshape(-1)[rp[eo[e]:eo[e + 1]]]
        assert np.all(held == e)


def test_noplan_rejects_batches_above_its_limit():
    T, k, E, G = 2049, 8, 256, 8
    L = moe.Layout(T, k, E, G)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ids = torch.zeros(T, k, dtype=torch.int32, device="cuda")
    w = torch.zeros(T, k, dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoEError) as ex:
        moe.moe_route_layout_noplan(ids, w, L, st)
    assert ex.value.code == moe.MOE_ERR_UNSUPPORTED


def test_noplan_path_combines_to_the_counting_sort_paths_output():
    cfg = inputs.MoEConfig("np_e2e", T=256, H=1024, E=64, G=8, k=8, N=512, zipf=1.2, seed=4)
    ids, w = gu.routed(cfg)
    x = inputs.make_x(cfg.T, cfg.H, cfg.seed).cuda()
    W = inputs.make_weights(cfg.E, cfg.N, cfg.H, cfg.seed).cuda()
    Wq = torch.empty(cfg.E, cfg.N, cfg.H, dtype=torch.uint8, device="cuda")
    Ws = torch.empty(cfg.E, cfg.N // 128, cfg.H // 128, dtype=torch.float32, device="cuda")
    moe.moe_quant_weights(W, Wq, Ws)
    R = cfg.T * cfg.k
    outs = []
    for noplan in (False, True):
        if noplan:
            L, st = noplan_layout(ids, w, cfg.E, cfg.G)
        else:
            L, st = gu.gpu_layout(ids, w, cfg.E, cfg.G)
        A = torch.empty(R, cfg.H, dtype=torch.uint8, device="cuda")
        As = torch.empty(cfg.H // 128, R, dtype=torch.float32, device="cuda")
        Y = torch.empty(R, cfg.N, dtype=torch.bfloat16, device="cuda")
        out = torch.empty(cfg.T, cfg.N, dtype=torch.bfloat16, device="cuda")
        moe.moe_dispatch_quant(x, L, A, As, st)
        moe.moe_grouped_gemm1(A, As, Wq, Ws, L, Y, st)
        moe.moe_combine(Y, L, out, st)
        torch.cuda.synchronize()
        assert st.item() == 0
        outs.append((gu.bits(out), gu.bits(Y), L["pair_row"].cpu().numpy()))
    (o0, y0, pr0), (o1, y1, pr1) = outs
    assert np.array_equal(y0[pr0], y1[pr1])       # each pair's GEMM1 row, wherever it was placed
    assert np.array_equal(o0, o1)
