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
