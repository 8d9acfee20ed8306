"""bnb_int8_linear_opts: the per-call options of benchmarks and tests (GPU).

- BNB_OPT_LEGACY_MMA: the warp-level mma GEMM, against the oracle, in every
  form (fp16 with W16, a bias, the int8 weight alone, bf16);
- BNB_OPT_MAIN_ONLY and BNB_OPT_NO_PDL change how the call is launched, not
  what it computes: Y is bit-identical to the plain call's;
- BNB_OPT_SINGLE_CTA: the 128 x 256 tile on single CTAs instead of the
  256 x 256 tile on CTA pairs (the default for T > 32): the same int32
  accumulators and Y bit for bit, and both match the oracle;
- BNB_OPT_FORCE_TIMEOUT: the main kernel takes its timeout path, the host
  reads BNB_ERR_TIMEOUT through bnb_last_device_status, and the next call on
  the same workspace (and context) runs normally and matches the oracle.
  The wait that gives up is on an mbarrier that nothing completes, with a
  limit of about 0.1 ms; nothing faults, traps or hangs.
"""

import math

import numpy as np
import pytest

import inputs
from parity import check_y, run_and_compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from int8_mixed_precision_04_b300 import binding, build
    build.build()
    binding.load()


SHAPES = [(17, 272, 129, 3), (300, 1024, 200, 4), (257, 2064, 1000, 7), (130, 512, 257, 40)]


@pytest.mark.parametrize("T,K,N,ncols", SHAPES)
@pytest.mark.parametrize("tau", [6.0, 0.0, math.inf])
def test_legacy_mma_fp16(orc, T, K, N, ncols, tau):
    from int8_mixed_precision_04_b300 import binding
    w = inputs.random_small(T, K, N, ncols, seed=T + 11 * N + K, tau=tau)
    run_and_compare(orc, w.X, w.W, tau, what=f"mma T{T} K{K} N{N} tau{tau}",
                    opts=binding.OPT_LEGACY_MMA)


@pytest.mark.parametrize("T,K,N,ncols", SHAPES[:3])
@pytest.mark.parametrize("form", ["bias", "wq_only"])
def test_legacy_mma_forms(orc, T, K, N, ncols, form):
    import torch

    from int8_mixed_precision_04_b300 import binding
    w = inputs.random_small(T, K, N, ncols, seed=T + 13 * N + K, tau=6.0)
    b = inputs.bias(N, K, seed=N)
    W = torch.from_numpy(w.W).cuda()
    Wq, sw = binding.quantize_weight(W)
    Y = binding.linear_opts(torch.from_numpy(w.X).cuda(), Wq, sw,
                            None if form == "wq_only" else W, 6.0, binding.OPT_LEGACY_MMA,
                            bias=torch.from_numpy(b).cuda())
    Wq_o, sw_o = orc.quantize_weight(w.W)
    ref = orc.linear(w.X, Wq_o, sw_o, None if form == "wq_only" else w.W, 6.0, bias=b)
    check_y(Y.cpu().numpy(), ref["Y"], f"mma {form} T{T} K{K} N{N}")


@pytest.mark.parametrize("T,K,N,ncols", SHAPES[:3])
@pytest.mark.parametrize("form", ["w16", "bias", "wq_only"])
def test_legacy_mma_bf16(orc, T, K, N, ncols, form):
    from int8_mixed_precision_04_b300 import binding
    from test_gpu_bf16 import _bf16_bits, _workload, run_bf16
    Xb, Wb = _workload(T, K, N, ncols, seed=T + 7 * N + K, tau=6.0)
    bias = _bf16_bits(inputs.bias(N, K, seed=N).astype(np.float32)) if form != "w16" else None
    run_bf16(orc, Xb, Wb, 6.0, bias=bias, wq_only=form == "wq_only",
             what=f"mma bf16 {form} T{T} K{K} N{N}", opts=binding.OPT_LEGACY_MMA)


@pytest.mark.parametrize("T,K,N", [(16, 4096, 4096), (5, 1040, 520), (300, 1024, 200),
                                   (2048, 4096, 1024)])
def test_launch_options_keep_results(T, K, N):
    """MAIN_ONLY after a full call on the same workspace, and NO_PDL, give
    the plain call's Y bit for bit."""
    import torch

    from int8_mixed_precision_04_b300 import binding
    w = inputs.random_small(T, K, N, 5, seed=T + K + N, tau=6.0)
    X = torch.from_numpy(w.X).cuda()
    W = torch.from_numpy(w.W).cuda()
    Wq, sw = binding.quantize_weight(W)
    ws = torch.empty(binding.workspace_bytes(T, N, K), dtype=torch.uint8, device="cuda")
    Y0 = binding.linear(X, Wq, sw, W, 6.0, workspace=ws)
    Y1 = binding.linear_opts(X, Wq, sw, W, 6.0, binding.OPT_MAIN_ONLY, workspace=ws)
    Y2 = binding.linear_opts(X, Wq, sw, W, 6.0, binding.OPT_NO_PDL, workspace=ws)
    Y3 = binding.linear_opts(X, Wq, sw, W, 6.0, binding.OPT_MAIN_ONLY | binding.OPT_NO_PDL,
                             workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(Y0, Y1) and torch.equal(Y0, Y2) and torch.equal(Y0, Y3)
    assert binding.last_device_status(ws) == 0


@pytest.mark.parametrize("T,K,N,ncols", [(33, 256, 100, 3), (40, 272, 129, 3), (300, 1024, 200, 4),
                                         (257, 2064, 1000, 7), (130, 512, 257, 40)])
@pytest.mark.parametrize("tau", [6.0, 0.0])
def test_cta_pair_and_single_cta_agree(orc, T, K, N, ncols, tau):
    """Both tile forms sum each output over K in the same order: identical
    accumulators and Y.  The single-CTA form also against the oracle (the
    pair form is what every other parity test runs for T > 32)."""
    import torch

    from int8_mixed_precision_04_b300 import binding
    w = inputs.random_small(T, K, N, ncols, seed=5 * T + N + K, tau=tau)
    r1, _ = run_and_compare(orc, w.X, w.W, tau, what=f"single-CTA T{T} K{K} N{N} tau{tau}",
                            opts=binding.OPT_SINGLE_CTA)
    X = torch.from_numpy(w.X).cuda()
    W = torch.from_numpy(w.W).cuda()
    Wq, sw = binding.quantize_weight(W)
    r2 = binding.linear_debug(X, Wq, sw, W, tau)
    torch.cuda.synchronize()
    assert binding.last_device_status(r2["workspace"]) == 0
    assert torch.equal(r1["acc"], r2["acc"]) and torch.equal(r1["Y"], r2["Y"])


@pytest.mark.parametrize("T,K,N,form", [(16, 4096, 4096, ""), (3, 272, 129, ""), (300, 1024, 200, ""),
                                        (2048, 4096, 1024, ""), (300, 1024, 200, "single_cta"),
                                        (9, 8192, 300, "")])
def test_forced_timeout_then_normal_call(orc, T, K, N, form):
    """A wait that gives up is reported through the status word, and the
    context and workspace stay usable: the next call is correct."""
    import torch

    from int8_mixed_precision_04_b300 import binding
    w = inputs.random_small(T, K, N, 4, seed=3 * T + K + N, tau=6.0)
    X = torch.from_numpy(w.X).cuda()
    W = torch.from_numpy(w.W).cuda()
    Wq, sw = binding.quantize_weight(W)
    ws = torch.empty(binding.workspace_bytes(T, N, K), dtype=torch.uint8, device="cuda")
    opts = binding.OPT_SINGLE_CTA if form == "single_cta" else 0
    binding.linear_opts(X, Wq, sw, W, 6.0, binding.OPT_FORCE_TIMEOUT | opts, workspace=ws)
    assert binding.last_device_status(ws) == binding.Status.TIMEOUT
    # the status word was read and cleared; the same workspace, a normal call
    Y = binding.linear(X, Wq, sw, W, 6.0, workspace=ws)
    assert binding.last_device_status(ws) == 0
    Wq_o, sw_o = orc.quantize_weight(w.W)
    rows = np.array(sorted({0, T - 1, T // 2}), dtype=np.int64)
    ref = orc.linear(w.X, Wq_o, sw_o, w.W, 6.0, rows=rows)
    check_y(Y.cpu().numpy()[rows], ref["Y"], f"after a forced timeout T{T} K{K} N{N}")


def test_unknown_options_are_rejected():
    import torch

    from int8_mixed_precision_04_b300 import binding
    X = torch.zeros((4, 64), dtype=torch.float16, device="cuda")
    W = torch.zeros((32, 64), dtype=torch.float16, device="cuda")
    Wq, sw = binding.quantize_weight(W)
    for bad in (0x80, binding.OPT_CLUSTER(3), binding.OPT_CLUSTER(32),
                binding.OPT_MAIN_ONLY | binding.OPT_ACT_ONLY):
        with pytest.raises(binding.BnbError) as e:
            binding.linear_opts(X, Wq, sw, W, 6.0, bad)
        assert e.value.status == binding.Status.INVALID_ARG
