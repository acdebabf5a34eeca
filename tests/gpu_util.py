"""Helpers shared by the GPU parity tests (not a test module).

Every expected value comes from the CPU oracle run on the same seeded inputs;
nothing here is computed by the CUDA path except what is being checked."""
from __future__ import annotations

import numpy as np
import torch

import combine_counting_sort_gb300 as moe
import oracle
from combine_counting_sort_gb300 import inputs

# Tolerance of the bf16 outputs of GEMM1 and combine against the oracle:
# max |y - y_ref| / max |y_ref| <= 1e-2 and ||y - y_ref||_2 / ||y_ref||_2 <= 5e-3.
MAX_REL, NORM_REL = 1e-2, 5e-3


def build():
    from combine_counting_sort_gb300 import _build
    _build.build()
    moe.lib()


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns on the host."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def assert_close_bf16(got_bits: np.ndarray, want_bits: np.ndarray, what: str):
    got = oracle.bf16_to_f32(got_bits).astype(np.float64)
    want = oracle.bf16_to_f32(want_bits).astype(np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    scale = np.max(np.abs(want))
    err = np.abs(got - want)
    max_rel = err.max() / scale if scale > 0 else err.max()
    norm = np.linalg.norm(want)
    norm_rel = np.linalg.norm(got - want) / norm if norm > 0 else np.linalg.norm(got - want)
    assert max_rel <= MAX_REL and norm_rel <= NORM_REL, f"{what}: max_rel {max_rel:.3e} norm_rel {norm_rel:.3e}"
    return max_rel, norm_rel


def routed(cfg: inputs.MoEConfig):
    """Top-k pairs from the oracle router on the config's seeded logits."""
    logits = inputs.make_logits(cfg.T, cfg.E, cfg.zipf, cfg.seed).numpy()
    return oracle.router_topk(logits, cfg.k)


def routing_with_counts(counts, seed=0):
    """k = 1 routing whose expert e receives exactly counts[e] tokens, in a
    seeded random token order; weights 1."""
    ids = np.repeat(np.arange(len(counts), dtype=np.int32), counts)
    np.random.default_rng(seed).shuffle(ids)
    return ids[:, None].copy(), np.ones((len(ids), 1), np.float32)


# Expert sizes around every boundary of the GEMM1 tile kinds: 1..32 rows
# (transposed), 33..64 and 65..127 (short A boxes), 128 and more, and the last
# tile of a larger expert on either side of 32 rows (160, 161).
FEW_ROW_COUNTS = [1, 2, 7, 8, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 159, 160, 161, 0, 5, 3, 300, 30]


def gpu_layout(ids: np.ndarray, w: np.ndarray, E: int, G: int):
    T, k = ids.shape
    L = moe.Layout(T, k, E, G)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_route_layout(torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), L, status)
    torch.cuda.synchronize()
    return L, status


def compare_layout(L: moe.Layout, ref: dict):
    got = L.numpy()
    for name, g in got.items():
        want = ref[name]
        if name == "row_weight":
            assert np.array_equal(g.view(np.uint32), np.asarray(want, np.float32).view(np.uint32)), name
        else:
            assert np.array_equal(g, np.asarray(want)), f"{name} differs"


# ---------------------------------------------------------------- MX scale-factor layouts
# The MX variant stores its e8m0 codes in 512-byte atoms: byte
# (i % 32) * 16 + (i // 32) * 4 + j of an atom holds row i's code of 32-value
# chunk j of one 128-value K block (the layout stated in include/moe.h).  These
# read the codes back per row, so they compare with the oracle's [rows, H/32].

def _atom_byte(i):
    i = np.asarray(i, dtype=np.int64)
    return (i % 32) * 16 + (i // 32) * 4


def sf_a_rows(A_sf: np.ndarray, ref: dict, rows: np.ndarray) -> np.ndarray:
    """A_sf [max_tiles, H/128, 512] -> e8m0 codes [len(rows), H/32] of dense rows
    ``rows``, placed by the oracle layout's tile of each row."""
    rows = np.asarray(rows, dtype=np.int64)
    eo = np.asarray(ref["expert_offset"], np.int64)
    eto = np.asarray(ref["expert_tile_offset"], np.int64)
    e = np.searchsorted(eo, rows, side="right") - 1
    rel = rows - eo[e]
    m, i = eto[e] + rel // 128, rel % 128
    KB = A_sf.shape[1]
    idx = _atom_byte(i)[:, None, None] + np.arange(4)[None, None, :]              # [n, 1, 4]
    out = A_sf[m[:, None, None], np.arange(KB)[None, :, None], idx]                 # [n, KB, 4]
    return out.reshape(len(rows), KB * 4)


def sf_w_rows(W_sf: np.ndarray, e: int, n_rows: np.ndarray) -> np.ndarray:
    """W_sf [E, H/128, N/128, 512] -> e8m0 codes [len(n_rows), H/32] of expert e's rows."""
    n_rows = np.asarray(n_rows, dtype=np.int64)
    KB = W_sf.shape[1]
    idx = _atom_byte(n_rows % 128)[:, None, None] + np.arange(4)[None, None, :]
    out = W_sf[e][np.arange(KB)[None, :, None], (n_rows // 128)[:, None, None], idx]
    return out.reshape(len(n_rows), KB * 4)
