"""GPU parity of the routing layout and the router helper against the oracle
(bit-exact tables), on the workloads' shapes and on edge cases."""
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


@pytest.mark.parametrize("name", ["tiny", "t2048_uniform", "t8192_zipf1.2", "stage1_t16384_zipf1.0"])
def test_layout_matches_oracle_on_workloads(name):
    cfg = inputs.CONFIGS[name]
    ids, w = gu.routed(cfg)
    L, status = gu.gpu_layout(ids, w, cfg.E, cfg.G)
    assert status.item() == 0
    gu.compare_layout(L, oracle.route_layout(ids, w, cfg.E, cfg.G))


@pytest.mark.parametrize("T,k,E,G,mode", [
    (1, 1, 1, 1, "uniform"), (3, 2, 4, 2, "uniform"), (37, 4, 16, 4, "dup"), (500, 6, 64, 8, "one_expert"),
    (1000, 32, 1024, 4, "uniform"), (129, 8, 256, 8, "skew"), (100000, 8, 256, 8, "skew"),
    (70000, 1, 3, 1, "uniform"),
    # either side of the single-block (plain launch) limit of 32 tokens
    (32, 8, 256, 8, "skew"), (33, 8, 256, 8, "skew"), (32, 32, 64, 4, "uniform"),
])
def test_layout_edge_cases(T, k, E, G, mode):
    rng = np.random.default_rng(T + k + E)
    if mode == "one_expert":
        ids = np.tile(np.arange(k, dtype=np.int32), (T, 1))      # every token to experts 0..k-1
    elif mode == "dup":
        ids = rng.integers(0, E, size=(T, k)).astype(np.int32)   # duplicate ids within tokens
    elif mode == "skew":
        p = 1.0 / np.arange(1, E + 1) ** 1.5
        ids = np.stack([rng.choice(E, size=k, replace=False, p=p / p.sum()) for _ in range(T)]).astype(np.int32)
    else:
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    L, status = gu.gpu_layout(ids, w, E, G)
    assert status.item() == 0
    gu.compare_layout(L, oracle.route_layout(ids, w, E, G))


def test_layout_back_to_back_calls_reuse_workspace():
    cfg = inputs.CONFIGS["t2048_uniform"]
    ids, w = gu.routed(cfg)
    L = moe.Layout(cfg.T, cfg.k, cfg.E, cfg.G)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ids_d, w_d = torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
    ref = oracle.route_layout(ids, w, cfg.E, cfg.G)
    for _ in range(3):
        for t in L.t.values():
            t.fill_(-7)                                   # poison: every entry must be rewritten
        moe.moe_route_layout(ids_d, w_d, L, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    gu.compare_layout(L, ref)


def test_layout_invalid_expert_id_is_reported():
    ids = np.array([[0, 1], [5, 2], [3, -1]], dtype=np.int32)
    w = np.ones((3, 2), np.float32)
    L, status = gu.gpu_layout(ids, w, 4, 2)
    assert status.item() == moe.MOE_ERR_EXPERT_ID
    pr = L["pair_row"].cpu().numpy()
    assert pr[2] == -1 and pr[5] == -1
    valid = [0, 1, 3, 4]
    assert sorted(pr[valid]) == [0, 1, 2, 3]


def layout_of_valid_pairs(ids, w, E, G):
    """The layout of the pairs with an id in [0, E), the others skipped: the
    oracle's definition (stable counting sort by (group, expert)) restricted
    to the valid pairs, each token's first expert taken over its valid ids."""
    T, k = ids.shape
    flat = ids.reshape(-1).astype(np.int64)
    ok = (flat >= 0) & (flat < E)
    epg = E // G
    p_valid = np.nonzero(ok)[0]
    key = (flat[p_valid] // epg) * E + flat[p_valid]
    row_pair = p_valid[np.argsort(key, kind="stable")]
    pair_row = np.full(T * k, -1, np.int64)
    pair_row[row_pair] = np.arange(len(row_pair))
    count = np.bincount(flat[ok], minlength=E)
    masked = np.where(ok.reshape(T, k), ids, E)
    first = masked.min(axis=1)
    has = first < E
    tok = np.nonzero(has)[0]
    token_order = tok[np.argsort(first[has], kind="stable")]
    return dict(pair_row=pair_row, row_pair=row_pair, row_weight=w.reshape(-1)[row_pair], count=count,
                expert_offset=np.concatenate([[0], np.cumsum(count)]),
                ready_tokens=np.cumsum(np.bincount(first[has], minlength=E)), token_order=token_order)


@pytest.mark.parametrize("T,k,E,G", [
    (20, 4, 16, 2),        # one block, plain launch
    (3000, 4, 32, 4),      # the grid, one staged chunk per block
    (80000, 8, 64, 8),     # the grid, several staged chunks per block
])
def test_layout_skips_and_reports_invalid_ids_at_every_grid_shape(T, k, E, G):
    rng = np.random.default_rng(T)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    bad = rng.random(ids.shape) < 0.01
    ids[bad] = np.where(rng.random(int(bad.sum())) < 0.5, -1, E + rng.integers(0, 4, int(bad.sum())))
    ids[0, 0] = E                                  # at least one of each kind
    ids[-1, -1] = -1
    w = rng.random((T, k)).astype(np.float32)
    L, status = gu.gpu_layout(ids, w, E, G)
    assert status.item() == moe.MOE_ERR_EXPERT_ID
    want = layout_of_valid_pairs(ids, w, E, G)
    got = L.numpy()
    n = len(want["row_pair"])
    assert np.array_equal(got["pair_row"], want["pair_row"])
    assert np.array_equal(got["row_pair"][:n], want["row_pair"])
    assert np.array_equal(got["row_weight"][:n].view(np.uint32), want["row_weight"].view(np.uint32))
    assert np.array_equal(got["count"], want["count"])
    assert np.array_equal(got["expert_offset"], want["expert_offset"])
    assert np.array_equal(got["ready_tokens"], want["ready_tokens"])
    assert np.array_equal(got["token_order"][: len(want["token_order"])], want["token_order"])


@pytest.mark.parametrize("T,E,k,zipf", [(128, 8, 2, None), (2048, 256, 8, None), (4096, 256, 8, 1.2),
                                        (300, 1024, 16, None), (64, 40, 32, None)])
def test_router_matches_oracle(T, E, k, zipf):
    logits = inputs.make_logits(T, E, zipf, seed=1)
    ids_ref, w_ref = oracle.router_topk(logits.numpy(), k)
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    moe.moe_router_topk(logits.cuda(), k, ids, w)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert np.allclose(w.cpu().numpy(), w_ref, rtol=2e-6, atol=1e-7)


def test_router_ties_go_to_lower_id():
    logits = torch.zeros(4, 16)
    logits[:, 3] = logits[:, 9] = 2.0
    ids = torch.empty(4, 3, dtype=torch.int32, device="cuda")
    w = torch.empty(4, 3, dtype=torch.float32, device="cuda")
    moe.moe_router_topk(logits.cuda(), 3, ids, w)
    ids_ref, _ = oracle.router_topk(logits.numpy(), 3)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert list(ids_ref[0]) == [3, 9, 0]
