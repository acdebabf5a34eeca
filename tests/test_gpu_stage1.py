"""GPU parity of the fused stage1 (quant + dispatch + GEMM1 overlapped through
per-tile / per-expert ready flags) against the oracle and against the unfused
calls: the fused kernel runs the same arithmetic in the same order, so its
A, A_scale and Y must be bit-identical to moe_dispatch_quant followed by
moe_grouped_gemm1, for every flag granularity, schedule and SM split.  Also
the bounded wait: a withheld tile makes the consumer give up with
MOE_ERR_TIMEOUT, and the context stays usable."""
import itertools

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


class Problem:
    def __init__(self, cfg, W=None):
        self.cfg = cfg
        self.x = inputs.make_x(cfg.T, cfg.H, cfg.seed).cuda()
        self.ids, self.w = gu.routed(cfg)
        self.L, st = gu.gpu_layout(self.ids, self.w, cfg.E, cfg.G)
        assert st.item() == 0
        if W is None:
            W = inputs.make_weights(cfg.E, cfg.N, cfg.H, cfg.seed, device="cuda")
        self.Wq = torch.empty(cfg.E, cfg.N, cfg.H, dtype=torch.uint8, device="cuda")
        self.Ws = torch.empty(cfg.E, cfg.N // 128, cfg.H // 128, dtype=torch.float32, device="cuda")
        moe.moe_quant_weights(W, self.Wq, self.Ws)
        self.R = cfg.T * cfg.k
        self.ws = torch.empty(int(self.L.sizes.stage1_ws_bytes), dtype=torch.uint8, device="cuda")
        # unfused reference outputs
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.A0, self.As0, self.Y0 = self.buffers()
        moe.moe_dispatch_quant(self.x, self.L, self.A0, self.As0, self.status)
        moe.moe_grouped_gemm1(self.A0, self.As0, self.Wq, self.Ws, self.L, self.Y0, self.status)
        torch.cuda.synchronize()
        assert self.status.item() == 0

    def buffers(self):
        cfg = self.cfg
        A = torch.full((self.R, cfg.H), 0x7F, dtype=torch.uint8, device="cuda")
        As = torch.full((cfg.H // 128, self.R), float("nan"), dtype=torch.float32, device="cuda")
        Y = torch.full((self.R, cfg.N), float("nan"), dtype=torch.bfloat16, device="cuda")
        return A, As, Y

    def fused(self, opts):
        A, As, Y = self.buffers()
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        moe.moe_stage1(self.x, self.L, self.Wq, self.Ws, A, As, Y, self.ws, status, opts)
        torch.cuda.synchronize()
        return A, As, Y, status.item()

    def check_same_as_unfused(self, opts):
        A, As, Y, st = self.fused(opts)
        assert st == 0, moe.status_string(st)
        assert torch.equal(A, self.A0)
        assert torch.equal(As.view(torch.int32), self.As0.view(torch.int32))
        assert torch.equal(Y.view(torch.int16), self.Y0.view(torch.int16))


@pytest.fixture(scope="module")
def small():
    cfg = inputs.MoEConfig("small_skew", T=600, H=512, E=32, G=4, k=4, N=512, zipf=1.2, seed=4)
    return Problem(cfg)


def test_stage1_tiny_matches_oracle():
    cfg = inputs.CONFIGS["tiny"]
    W = inputs.make_weights(cfg.E, cfg.N, cfg.H, cfg.seed)
    P = Problem(cfg, W.cuda())
    A, As, Y, st = P.fused(moe.stage1_opts(comm_sms=2))
    assert st == 0
    q, s = oracle.quantize_rows(inputs.bf16_bits(P.x.cpu()))
    A_ref, As_ref = oracle.dispatch(q, s, P.L["pair_row"].cpu().numpy(), cfg.k)
    assert np.array_equal(A.cpu().numpy(), A_ref)
    assert np.array_equal(As.cpu().numpy().view(np.uint32), As_ref.view(np.uint32))
    Wq, Ws = oracle.quantize_weights(inputs.bf16_bits(W))
    Y_ref = oracle.grouped_gemm1(A_ref, As_ref, Wq, Ws, P.L["expert_offset"].cpu().numpy())
    gu.assert_close_bf16(gu.bits(Y), Y_ref, "stage1 Y")


@pytest.mark.parametrize("flags,schedule,join,comm", list(itertools.product(
    [moe.MOE_FLAGS_PER_TILE, moe.MOE_FLAGS_PER_EXPERT], [moe.MOE_SCHED_EXPERT_MAJOR, moe.MOE_SCHED_READY_FIRST],
    [0, 1], [8, 36])))
def test_stage1_option_matrix_bit_identical_to_unfused(small, flags, schedule, join, comm):
    small.check_same_as_unfused(moe.stage1_opts(comm_sms=comm, flags=flags, schedule=schedule,
                                                producers_join=join))


@pytest.mark.parametrize("comm", [1, 16, 24])
def test_stage1_comm_sm_counts(small, comm):
    small.check_same_as_unfused(moe.stage1_opts(comm_sms=comm))


def test_stage1_wide_rows():
    # H = 8192: two staging rows per producer warp no longer fit in the idle
    # stage buffers, so the producers store code rows directly instead of by
    # bulk copies; the result is the same
    cfg = inputs.MoEConfig("wide", T=300, H=8192, E=8, G=2, k=4, N=256, zipf=1.2, seed=9)
    P = Problem(cfg)
    for opts in (moe.stage1_opts(comm_sms=8), moe.stage1_opts(comm_sms=24, schedule=moe.MOE_SCHED_READY_FIRST)):
        P.check_same_as_unfused(opts)


def test_stage1_k12_bit_identical_to_unfused():
    # k > 8: the producers' block scales go out in two groups of 8 rows
    cfg = inputs.MoEConfig("k12", T=400, H=512, E=48, G=4, k=12, N=256, zipf=1.1, seed=12)
    P = Problem(cfg)
    for opts in (moe.stage1_opts(comm_sms=8), moe.stage1_opts(comm_sms=24, flags=moe.MOE_FLAGS_PER_EXPERT)):
        P.check_same_as_unfused(opts)


def test_stage1_full_size_bit_identical_to_unfused():
    # the benchmark's step configuration and two others at T=8192
    P = Problem(inputs.CONFIGS["t8192_zipf1.2"])
    for opts in (moe.stage1_opts(), moe.stage1_opts(comm_sms=24, schedule=moe.MOE_SCHED_READY_FIRST),
                 moe.stage1_opts(comm_sms=8, flags=moe.MOE_FLAGS_PER_EXPERT, producers_join=0)):
        P.check_same_as_unfused(opts)


def test_stage1_t16384_sweep_configurations_bit_identical_to_unfused():
    # the fused-stage1 sweep's workload (T=16384, Zipf 1.0): every producer SM
    # count it times, across both flag granularities and both schedules
    P = Problem(inputs.CONFIGS["stage1_t16384_zipf1.0"])
    for comm, flags, schedule in [(8, moe.MOE_FLAGS_PER_TILE, moe.MOE_SCHED_EXPERT_MAJOR),
                                  (16, moe.MOE_FLAGS_PER_EXPERT, moe.MOE_SCHED_READY_FIRST),
                                  (24, moe.MOE_FLAGS_PER_TILE, moe.MOE_SCHED_READY_FIRST),
                                  (36, moe.MOE_FLAGS_PER_EXPERT, moe.MOE_SCHED_EXPERT_MAJOR),
                                  (36, moe.MOE_FLAGS_PER_TILE, moe.MOE_SCHED_EXPERT_MAJOR)]:
        P.check_same_as_unfused(moe.stage1_opts(comm_sms=comm, flags=flags, schedule=schedule))


@pytest.mark.parametrize("schedule", [moe.MOE_SCHED_EXPERT_MAJOR, moe.MOE_SCHED_READY_FIRST])
def test_stage1_withheld_tile_times_out_and_context_survives(small, schedule):
    opts = moe.stage1_opts(comm_sms=8, schedule=schedule, timeout_ns=20_000_000, withhold_tile=0)
    A, As, Y, st = small.fused(opts)
    assert st == moe.MOE_ERR_TIMEOUT
    # the next call on the same context is clean
    small.check_same_as_unfused(moe.stage1_opts(comm_sms=8, schedule=schedule))
