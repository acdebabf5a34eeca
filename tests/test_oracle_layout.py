"""Pins for the oracle's router and routing layout.

Layout: a hand-worked fixture, brute force with Python's ``sorted`` on tiny
inputs, and the invariants the mori stage1 page fixes (every token appears k
times, counts sum to T*k, a landed prefix of the token order completes a prefix
of the experts).  Router: brute force, torch's softmax + topk (library), and
properties of renormalised softmax weights."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from combine_counting_sort_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_layout_handworked_fixture():
    with open(os.path.join(GOLDEN, "layout_handworked.json")) as f:
        g = json.load(f)
    out = oracle.route_layout(np.array(g["topk_ids"], np.int32), np.array(g["topk_w"], np.float32),
                              g["E"], g["G"], g["block_m"])
    for name, want in g["expected"].items():
        if name == "max_tiles":
            assert out[name] == want
        elif name == "row_weight":
            assert np.array_equal(out[name], np.array(want, np.float32)), name
        else:
            assert np.array_equal(out[name], np.array(want)), name


def brute_layout(ids, E, G, BM):
    """Tables by direct enumeration: Python sort of (group, expert, pair) triples."""
    T, k = ids.shape
    epg = E // G
    triples = sorted((int(ids[t, j]) // epg, int(ids[t, j]), t * k + j) for t in range(T) for j in range(k))
    row_pair = [p for _, _, p in triples]
    count = [sum(1 for _, e, _ in triples if e == x) for x in range(E)]
    rowmap, tile_expert, tile_rows = [], [], []
    r = 0
    for e in range(E):
        for i in range(math.ceil(count[e] / BM)):
            n = min(BM, count[e] - i * BM)
            rowmap += list(range(r, r + n)) + [-1] * (BM - n)
            tile_expert.append(e)
            tile_rows.append(n)
            r += n
    firsts = [min(int(x) for x in ids[t]) for t in range(T)]
    token_order = sorted(range(T), key=lambda t: (firsts[t], t))
    return row_pair, count, rowmap, tile_expert, tile_rows, token_order


@pytest.mark.parametrize("T,k,E,G,BM,seed", [
    (1, 1, 1, 1, 128, 0), (7, 3, 5, 5, 2, 1), (16, 4, 8, 2, 3, 2), (33, 2, 6, 3, 4, 3),
    (20, 4, 4, 1, 128, 4), (50, 8, 16, 4, 5, 5),
])
def test_layout_brute_force(T, k, E, G, BM, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)   # duplicates within a token allowed
    w = rng.random((T, k)).astype(np.float32)
    out = oracle.route_layout(ids, w, E, G, BM)
    row_pair, count, rowmap, tile_expert, tile_rows, token_order = brute_layout(ids, E, G, BM)
    nt = len(tile_expert)
    assert list(out["row_pair"]) == row_pair
    assert list(out["count"]) == count
    assert out["num_tiles"][0] == nt
    assert list(out["rowmap"][: nt * BM]) == rowmap
    assert np.all(out["rowmap"][nt * BM:] == -1)
    assert list(out["tile_expert"][:nt]) == tile_expert
    assert list(out["tile_rows"][:nt]) == tile_rows
    assert list(out["token_order"]) == token_order
    assert np.array_equal(out["row_weight"], w.reshape(-1)[row_pair])


def check_layout_invariants(ids, E, G, BM, out):
    T, k = ids.shape
    R = T * k
    flat = ids.reshape(-1)
    # every token appears exactly k times among the rows; counts sum to T*k
    assert np.array_equal(np.bincount(out["row_pair"] // k, minlength=T), np.full(T, k))
    assert out["count"].sum() == R
    # pair_row and row_pair are inverse permutations
    assert np.array_equal(np.sort(out["row_pair"]), np.arange(R))
    assert np.array_equal(out["pair_row"][out["row_pair"]], np.arange(R))
    # expert-major, and ascending (token, slot) within an expert
    eo = out["expert_offset"]
    for e in range(E):
        rows = out["row_pair"][eo[e]:eo[e + 1]]
        assert np.all(flat[rows] == e)
        assert np.all(np.diff(rows) > 0)
    # group runs are unions of consecutive experts
    assert np.array_equal(out["group_offset"], eo[np.arange(G + 1) * (E // G)])
    # tiles: rows per tile within the sort block, all rows covered once by the rowmap
    nt = out["num_tiles"][0]
    assert nt <= out["max_tiles"]
    tr = out["tile_rows"]
    assert tr[:nt].sum() == R and np.all((tr[:nt] >= 1) & (tr[:nt] <= BM)) and np.all(tr[nt:] == 0)
    rm = out["rowmap"]
    assert np.array_equal(np.sort(rm[rm >= 0]), np.arange(R))
    for m in range(nt):
        e = out["tile_expert"][m]
        assert eo[e] <= out["tile_row_begin"][m] and out["tile_row_begin"][m] + tr[m] <= eo[e + 1]
    # landed prefix: once the first P tokens of token_order have landed, every
    # expert e with ready_tokens[e] <= P is complete, and those experts form a
    # prefix 0..e* of the expert order (a prefix of each group's experts)
    pos = np.empty(T, np.int64)
    pos[out["token_order"]] = np.arange(T)
    rt = out["ready_tokens"]
    assert np.all(np.diff(rt) >= 0) and rt[-1] == T
    for e in range(E):
        toks = np.nonzero((ids == e).any(axis=1))[0]
        assert np.all(pos[toks] < rt[e])
    for P in range(0, T + 1, max(1, T // 17)):
        done = np.nonzero(rt <= P)[0]
        assert np.array_equal(done, np.arange(len(done)))
        landed = np.zeros(T, bool)
        landed[out["token_order"][:P]] = True
        for e in done:
            assert landed[(ids == e).any(axis=1)].all()


@pytest.mark.parametrize("name", ["tiny", "t2048_uniform", "t8192_zipf1.2"])
def test_layout_invariants_on_workloads(name):
    cfg = inputs.CONFIGS[name]
    logits = inputs.make_logits(cfg.T, cfg.E, cfg.zipf, cfg.seed).numpy()
    # the layout only needs ids; take the k largest logits directly (same selection as the router)
    ids = np.argsort(-logits, axis=1, kind="stable")[:, : cfg.k].astype(np.int32)
    w = np.full(ids.shape, 1.0 / cfg.k, np.float32)
    out = oracle.route_layout(ids, w, cfg.E, cfg.G)
    check_layout_invariants(ids, cfg.E, cfg.G, oracle.BLOCK, out)
    if cfg.zipf is not None:
        # the skewed workload leaves experts empty and makes a few large
        assert (out["count"] == 0).sum() >= 1 and out["count"].max() > 1000


def test_max_tiles_bound_is_reached():
    # the capacity formula is tight: one expert with 1 + (T*k - (E-1)) rows and E-1 experts of 1 row
    T, k, E, BM = 40, 4, 8, 16
    R = T * k
    counts = [R - (E - 1)] + [1] * (E - 1)
    tiles = sum(math.ceil(c / BM) for c in counts)
    assert tiles <= oracle.max_tiles(T, k, E, BM)
    # brute force over all ways to split R pairs among E experts with per-expert residues
    best = 0
    for r in range(1, BM + 1):                # residues of 1 maximise padding
        rest = R - (E - 1) * r
        if rest > 0:
            best = max(best, (E - 1) * math.ceil(r / BM) + math.ceil(rest / BM))
    assert best <= oracle.max_tiles(T, k, E, BM)
    assert oracle.max_tiles(T, k, E, BM) - best <= 1


# ---------------------------------------------------------------- router

def test_router_brute_force_tiny():
    rng = np.random.default_rng(7)
    T, E, k = 40, 9, 3
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[3, 2] = logits[3, 5] = logits[3].max() + 1      # a tie at the top
    ids, w = oracle.router_topk(logits, k)
    for t in range(T):
        want = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))[:k]
        assert list(ids[t]) == want
    assert list(ids[3][:2]) == [2, 5]                       # tie: lower id first
    assert np.allclose(w.sum(axis=1), 1.0, atol=4e-7)
    assert np.all(np.diff(w, axis=1) <= 0)


def test_router_matches_torch_softmax_topk():
    logits = inputs.make_logits(256, 64, zipf=1.1, seed=3).numpy()
    ids, w = oracle.router_topk(logits, 6)
    p = torch.softmax(torch.from_numpy(logits).double(), dim=1)
    v, i = torch.topk(p, 6, dim=1)
    assert np.array_equal(ids, i.numpy())
    assert np.allclose(w, (v / v.sum(1, keepdim=True)).numpy(), rtol=1e-6, atol=0)


def test_router_weights_are_softmax_of_selected_logits():
    rng = np.random.default_rng(9)
    logits = rng.standard_normal((64, 32)).astype(np.float32)
    ids, w = oracle.router_topk(logits, 4)
    sel = np.take_along_axis(logits, ids, 1).astype(np.float64)
    # ratios of weights are exp of logit differences (the global softmax constant cancels)
    assert np.allclose(w[:, 1:] / w[:, :1], np.exp(sel[:, 1:] - sel[:, :1]), rtol=1e-6)
    # shift invariance
    ids2, w2 = oracle.router_topk(logits + np.float32(5.0), 4)
    assert np.array_equal(ids, ids2) and np.allclose(w, w2, rtol=1e-6)


# ---- per-(token, group) send runs (the next step of the path)

def brute_runs(ids, E, G):
    """Send rows by direct enumeration: Python sort of (group, first expert of
    the token in the group, token) over the tokens with a route into the group."""
    T, k = ids.shape
    epg = E // G
    keys = sorted((g, min(int(e) for e in ids[t] if int(e) // epg == g), t)
                  for t in range(T) for g in range(G) if any(int(e) // epg == g for e in ids[t]))
    send_row = {(t, g): s for s, (g, _, t) in enumerate(keys)}
    run_offset = [sum(1 for g2, _, _ in keys if g2 < g) for g in range(G + 1)]
    return keys, send_row, run_offset


@pytest.mark.parametrize("T,k,E,G,seed", [(1, 1, 1, 1, 0), (9, 3, 6, 3, 1), (25, 4, 8, 2, 2), (40, 6, 12, 4, 3),
                                         (30, 5, 5, 1, 4), (17, 4, 16, 16, 5)])
def test_group_runs_brute_force(T, k, E, G, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)           # duplicates allowed
    L = oracle.route_layout(ids, np.ones((T, k), np.float32), E, G)
    out = oracle.group_runs(ids, E, G, L["row_pair"])
    keys, send_row, run_offset = brute_runs(ids, E, G)
    assert list(out["run_offset"]) == run_offset
    assert list(out["send_token"]) == [t for _, _, t in keys]
    for t in range(T):
        for g in range(G):
            assert out["send_row"][t, g] == send_row.get((t, g), -1)
    epg = E // G
    for r, p in enumerate(L["row_pair"]):
        t, e = p // k, int(ids.reshape(-1)[p])
        assert out["gather_row"][r] == send_row[(t, e // epg)]


@pytest.mark.parametrize("name", ["tiny", "t2048_uniform", "t8192_zipf1.2"])
def test_group_runs_invariants_on_workloads(name):
    cfg = inputs.CONFIGS[name]
    logits = inputs.make_logits(cfg.T, cfg.E, cfg.zipf, cfg.seed).numpy()
    ids, w = oracle.router_topk(logits, cfg.k)
    L = oracle.route_layout(ids, w, cfg.E, cfg.G)
    out = oracle.group_runs(ids, cfg.E, cfg.G, L["row_pair"])
    epg = cfg.E // cfg.G
    grp = ids.astype(np.int64) // epg
    # one send row per (token, group) with a route into the group, and no other
    pairs = {(t, g) for t in range(cfg.T) for g in set(grp[t].tolist())}
    S = int(out["run_offset"][-1])
    assert S == len(pairs) == len(out["send_token"]) and S <= cfg.T * cfg.k
    assert sorted(out["send_row"][out["send_row"] >= 0].tolist()) == list(range(S))
    # every dense row gathers a send row of its own token
    tok_of_row = L["row_pair"] // cfg.k
    assert np.array_equal(out["send_token"][out["gather_row"]], tok_of_row)
    # a landed prefix of a run is a prefix of experts: every token routed to
    # expert e sits before run_ready[e] in its group's run
    for e in range(cfg.E):
        rows = out["gather_row"][L["expert_offset"][e]:L["expert_offset"][e + 1]]
        assert np.all(rows < out["run_ready"][e])
        assert np.all(rows >= out["run_offset"][e // epg])
    assert np.all(np.diff(out["run_ready"].reshape(cfg.G, epg), axis=1) >= 0)


def test_send_runs_gather_reproduces_the_dense_dispatch():
    # reading A through gather_row gives the dense dispatch buffer bit for bit
    cfg = inputs.MoEConfig("runs", T=300, H=512, E=32, G=4, k=6, N=256, zipf=1.2, seed=7)
    logits = inputs.make_logits(cfg.T, cfg.E, cfg.zipf, cfg.seed).numpy()
    ids, w = oracle.router_topk(logits, cfg.k)
    L = oracle.route_layout(ids, w, cfg.E, cfg.G)
    q, s = oracle.quantize_rows(inputs.bf16_bits(inputs.make_x(cfg.T, cfg.H, cfg.seed)))
    A, As = oracle.dispatch(q, s, L["pair_row"], cfg.k)
    R = oracle.group_runs(ids, cfg.E, cfg.G, L["row_pair"])
    A_send, As_send = oracle.dispatch_runs(q, s, R["send_token"])
    assert np.array_equal(A_send[R["gather_row"]], A)
    assert np.array_equal(As_send[:, R["gather_row"]].view(np.uint32), As.view(np.uint32))
    assert A_send.shape[0] < A.shape[0]
