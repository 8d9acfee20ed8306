"""CUDA path vs the oracle, element by element, through the C ABI (GPU)."""

import math

import numpy as np
import pytest

import inputs
from parity import run_and_compare, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from int8_mixed_precision_04_b300 import binding, build
    build.build()
    binding.load()


def test_tiny(orc):
    w = inputs.tiny()
    r, ref = run_and_compare(orc, w.X, w.W, w.tau, what="tiny")
    assert 7 in ref["O"] and 133 in ref["O"]


@pytest.mark.parametrize("T", inputs.DECODE_TS)
def test_decode(orc, T):
    w = inputs.decode(T=T)
    run_and_compare(orc, w.X, w.W, w.tau, what=f"decode T={T}")


@pytest.mark.parametrize("cluster", [16, 8, 4])
@pytest.mark.parametrize("T,K,N,ncols", [
    (16, 4096, 1024, 4), (5, 272, 200, 2), (16, 1040, 96, 70), (11, 2048, 520, 9),
    (16, 4096, 3900, 70),
])
def test_decode_cluster_sizes(orc, cluster, T, K, N, ncols):
    """The decode kernel with each cluster size it can run (16, 8 or 4 CTAs
    sharing one activation pass): CTAs with few or no columns, slices of up
    to 35 channels (a partial fifth 8-channel group), and more outlier columns
    than the producer warp sums alone.  A size whose resident CTAs cannot
    hold the call falls back to one that can."""
    from int8_mixed_precision_04_b300 import binding
    assert binding.load().bnb_int8_linear_path(T, N, K) == 1
    w = inputs.random_small(T, K, N, ncols, seed=K + N + cluster, tau=6.0)
    run_and_compare(orc, w.X, w.W, 6.0, what=f"decode cluster {cluster} T{T} K{K} N{N}",
                    opts=binding.OPT_CLUSTER(cluster))


@pytest.mark.parametrize("cluster", [1, 16, 8])
@pytest.mark.parametrize("T,K,N,ncols", [
    (1, 4096, 4096, 4), (8, 4096, 5900, 70), (2, 272, 200, 2), (7, 1040, 96, 70),
    (3, 2048, 520, 9), (8, 16, 1, 0), (4, 4096, 40, 12), (5, 4096, 4100, 1),
])
def test_decode_local(orc, cluster, T, K, N, ncols):
    """T <= 8 without clusters (every CTA runs the whole activation pass and
    takes up to three 16-channel weight tiles as A operands; BNB_OPT_CLUSTER(1),
    the default there), against the clustered kernel forced on the same
    shapes: slices of 8 to 40 channels (a partial last tile), K not a multiple
    of the warps' K-ranges, more outlier columns than the TMA boxes take, and
    N up to what the resident CTAs hold without clusters."""
    from int8_mixed_precision_04_b300 import binding
    assert binding.load().bnb_int8_linear_path(T, N, K) == 1
    assert binding.decode_cluster(T, N, K) == 1 if T <= (6 if K > 2048 else 5) else binding.decode_cluster(T, N, K) in (1, 4, 8, 16)
    w = inputs.random_small(T, K, N, ncols, seed=3 * K + N + T, tau=6.0)
    run_and_compare(orc, w.X, w.W, 6.0, what=f"decode local/cluster {cluster} T{T} K{K} N{N}",
                    opts=binding.OPT_CLUSTER(cluster))


@pytest.mark.parametrize("T", [1, 5, 16])
def test_decode_on_the_gemm(orc, T):
    """The decode workload through the tcgen05 GEMM's 32-token tile
    (BNB_OPT_GEMM), which a T <= 16 call otherwise takes only for weights the
    decode kernel cannot hold."""
    from int8_mixed_precision_04_b300 import binding
    w = inputs.decode(T=T)
    run_and_compare(orc, w.X, w.W, w.tau, what=f"decode on the GEMM T={T}", opts=binding.OPT_GEMM)


@pytest.mark.parametrize("T,K,N,ncols", [
    (1, 16, 1, 0), (3, 48, 7, 1), (16, 272, 129, 2), (17, 64, 300, 3), (33, 1040, 65, 4),
    (130, 512, 257, 5), (200, 2064, 131, 7), (257, 128, 1000, 2), (64, 4096, 64, 9),
])
@pytest.mark.parametrize("tau", [6.0, 3.0, 0.0, math.inf])
def test_ragged_shapes(orc, T, K, N, ncols, tau):
    w = inputs.random_small(T, K, N, ncols, seed=T * 7 + K + N, tau=tau)
    run_and_compare(orc, w.X, w.W, tau, what=f"T{T} K{K} N{N} tau{tau}")


@pytest.mark.parametrize("T,K,N,ncols,single", [
    (2049, 272, 300, 3, False), (2573, 64, 520, 2, False), (4100, 128, 257, 4, False),
    (2573, 64, 520, 2, True),
])
def test_token_tile_groups(orc, T, K, N, ncols, single):
    """The GEMM walks token tiles in groups of 8 (2048 tokens): a last group of
    one tile, a ragged last tile, a third group; every element against the
    oracle, on CTA pairs and (once) on single CTAs."""
    from int8_mixed_precision_04_b300 import binding
    w = inputs.random_small(T, K, N, ncols, seed=T + 3 * K + N, tau=6.0)
    run_and_compare(orc, w.X, w.W, 6.0, what=f"tile groups T{T} K{K} N{N}",
                    opts=binding.OPT_SINGLE_CTA if single else 0)


@pytest.mark.parametrize("T,K,N,ncols,tau", [
    (300, 1024, 200, 5, 6.0), (149, 4096, 96, 70, 6.0), (40, 2048, 64, 3, 0.0),
    (700, 512, 130, 40, 3.0), (17, 256, 300, 1, 6.0), (33, 16384, 64, 9, 6.0),
])
def test_act_pass_forms(orc, T, K, N, ncols, tau):
    """The GEMM path's activation pass: rows held in registers (K <= 8192) and
    read twice (K = 16384), sparse outlier blocks with the W16 gather, dense
    outlier blocks, and as many W16 rows as tokens or many more."""
    w = inputs.random_small(T, K, N, ncols, seed=T + K + ncols, tau=tau)
    run_and_compare(orc, w.X, w.W, tau, what=f"act pass T{T} K{K} tau{tau}")


@pytest.mark.parametrize("T", [5, 40])
def test_edge_rows(orc, T):
    """An all-zero row, a row whose every column is an outlier, a value exactly
    at the threshold, and zero weight rows."""
    w = inputs.random_small(T, 320, 96, 3, seed=99)
    X, W = w.X.copy(), w.W.copy()
    X[1] = 0
    X[2] = 9.0
    X[3, 10] = -6.0
    W[5] = 0
    run_and_compare(orc, X, W, 6.0, what="edge rows")


@pytest.mark.parametrize("T,K", [(16, 8192), (256, 8192), (48, 1024)])
@pytest.mark.parametrize("adversarial", [False, True])
def test_integer_inputs_exact(orc, T, K, adversarial):
    """tau = inf on integer inputs: codes equal the inputs and acc is the exact
    integer product, up to 127^2 * K in magnitude (1.3e8 at K = 8192)."""
    X, W = inputs.int_valued(T, K, 72, seed=5, adversarial=adversarial)
    r, ref = run_and_compare(orc, X, W, math.inf, what="integer inputs")
    if adversarial:
        assert np.abs(ref["acc"]).max() == 127 * 127 * K


@pytest.mark.parametrize("T", [16, 40])
def test_code_rounding_ties(orc, T):
    """Every code is an exact half-integer quotient: row absmax 127 * 2^e and
    values (k + 1/2) * 2^e, so 127 x / sx = k + 1/2 and the code must round to
    the even neighbour (the decode path at T = 16, the GEMM path at T = 40)."""
    rng = np.random.default_rng(17)
    K = 512
    X = np.empty((T, K), dtype=np.float64)
    for t in range(T):
        e = int(rng.integers(-9, 6))
        vals = (rng.integers(-127, 127, size=K) + 0.5) * 2.0 ** e
        vals[rng.integers(0, K)] = 127.0 * 2.0 ** e * (1 if t % 2 else -1)
        X[t] = vals
    X16 = X.astype(np.float16)
    assert np.array_equal(X16.astype(np.float64), X)  # every value exact in fp16
    W = (rng.standard_normal((96, K)) * 0.02).astype(np.float16)
    r, ref = run_and_compare(orc, X16, W, math.inf, what=f"ties T{T}")
    q = ref["Xq"].astype(np.int64)
    assert np.all(q % 2 == 0) or np.any(np.abs(q) == 127)  # ties went to even codes


def test_workspace_reuse(orc):
    """Consecutive calls on one workspace with different thresholds."""
    import torch

    from int8_mixed_precision_04_b300 import binding
    w = inputs.random_small(24, 256, 40, 4, seed=3)
    X = torch.from_numpy(w.X).cuda()
    W = torch.from_numpy(w.W).cuda()
    Wq, sw = binding.quantize_weight(W)
    ws = torch.empty(binding.workspace_bytes(24, 40, 256), dtype=torch.uint8, device="cuda")
    Wq_o, sw_o = orc.quantize_weight(w.W)
    for tau in (6.0, 0.0, math.inf, 3.0, 6.0):
        Y = binding.linear(X, Wq, sw, W, tau, workspace=ws)
        ref = orc.linear(w.X, Wq_o, sw_o, w.W, tau)
        from parity import check_y
        check_y(Y.cpu().numpy(), ref["Y"], f"reuse tau={tau}")


@pytest.mark.parametrize("T,K,N", [(16, 4096, 4096), (300, 1024, 200)])
def test_from_host(orc, T, K, N):
    """bnb_int8_linear_from_host (pinned host X in, pinned host Y out, on two
    streams in turn) gives the oracle's Y and exactly bnb_int8_linear's."""
    import torch

    from int8_mixed_precision_04_b300 import binding
    from parity import check_y
    w = inputs.random_small(T, K, N, 4, seed=T + N)
    W = torch.from_numpy(w.W).cuda()
    Wq, sw = binding.quantize_weight(W)
    Y_ref = binding.linear(torch.from_numpy(w.X).cuda(), Wq, sw, W, 6.0).cpu()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for i in range(4):
        Xh = torch.from_numpy(w.X).pin_memory()
        Yh = torch.empty((T, N), dtype=torch.float16).pin_memory()
        Xd = torch.empty((T, K), dtype=torch.float16, device="cuda")
        Yd = torch.empty((T, N), dtype=torch.float16, device="cuda")
        ws = torch.empty(binding.workspace_bytes(T, N, K), dtype=torch.uint8, device="cuda")
        binding.linear_from_host(Xh, Wq, sw, W, 6.0, Yh, Xd, Yd, ws, stream=streams[i % 2])
        outs.append((Yh, Xd, Yd, ws))
    torch.cuda.synchronize()
    Wq_o, sw_o = orc.quantize_weight(w.W)
    ref = orc.linear(w.X, Wq_o, sw_o, w.W, 6.0)
    for Yh, *_ in outs:
        assert torch.equal(Yh, Y_ref)
        check_y(Yh.numpy(), ref["Y"], f"from host T{T}")


@pytest.mark.parametrize("frac", inputs.SWEEP_FRACTIONS)
@pytest.mark.parametrize("tau", inputs.SWEEP_TAUS)
def test_sweep_reduced(orc, frac, tau):
    """The decomposition sweep's 16 points at a reduced size (K = N = 1024)."""
    w = inputs.sweep(frac, tau, T=512, K=1024, N=1024)
    run_and_compare(orc, w.X, w.W, tau, what=f"sweep-reduced f{frac} tau{tau}")


# ---- full sizes of the named workloads, on sampled rows --------------------

def test_prefill_full(orc):
    w = inputs.prefill()
    run_and_compare(orc, w.X, w.W, w.tau, rows=sample_rows(w.T), what="prefill")


def test_large_full(orc):
    w = inputs.large()
    run_and_compare(orc, w.X, w.W, w.tau, rows=sample_rows(w.T), what="large")


@pytest.mark.parametrize("frac", inputs.SWEEP_FRACTIONS)
@pytest.mark.parametrize("tau", inputs.SWEEP_TAUS)
def test_sweep_full(orc, frac, tau):
    w = inputs.sweep(frac, tau)
    run_and_compare(orc, w.X, w.W, tau, rows=sample_rows(w.T, 32), what=f"sweep f{frac} tau{tau}")


# ---- the decode path at every weight shape ---------------------------------

@pytest.mark.parametrize("T", [1, 16])
@pytest.mark.parametrize("K,N", [(4096, 11008), (8192, 28672)])
def test_decode_large_weights(orc, T, K, N):
    """A decode step (T <= 16) through the prefill and the large MLP weights,
    shapes the decode kernel's resident CTAs cannot hold (the tcgen05 GEMM
    takes them), every row and channel against the oracle."""
    w = inputs.decode(T=T, K=K, N=N)
    run_and_compare(orc, w.X, w.W, w.tau, what=f"decode T{T} K{K} N{N}")


@pytest.mark.parametrize("T,K,N,ncols", [
    (16, 4096, 5000, 4), (2, 4096, 6000, 70), (1, 4096, 17000, 3), (9, 2048, 9601, 9),
    (3, 272, 17000, 2),
])
def test_decode_several_launches(orc, T, K, N, ncols):
    """Channels beyond one wave of the decode kernel's resident CTAs: the
    call splits them over up to three launches (each with the activation
    pass), every element against the oracle."""
    import torch

    from int8_mixed_precision_04_b300 import binding
    lib = binding.load()
    assert lib.bnb_int8_linear_path(T, N, K) == 1
    w = inputs.random_small(T, K, N, ncols, seed=7 * K + N + T, tau=6.0)
    run_and_compare(orc, w.X, w.W, 6.0, what=f"decode, several launches, T{T} K{K} N{N}")
    # one call is more than one launch of the decode kernel, three at most
    X = torch.from_numpy(w.X).cuda()
    W = torch.from_numpy(w.W).cuda()
    Wq, sw = binding.quantize_weight(W)
    torch.cuda.synchronize()
    before = lib.bnb_launch_count()
    binding.linear(X, Wq, sw, W, 6.0)
    torch.cuda.synchronize()
    assert 2 <= lib.bnb_launch_count() - before <= 3


@pytest.mark.parametrize("T,K,N,ncols,tau", [
    (16, 1040, 3000, 6, 6.0), (7, 3072, 2056, 3, 6.0), (16, 8192, 1000, 40, 3.0),
    (2, 5120, 9000, 2, 6.0), (16, 2048, 40000, 5, 6.0), (9, 16, 37, 1, 0.0),
    (16, 6144, 777, 0, math.inf),
])
def test_decode_shapes(orc, T, K, N, ncols, tau):
    """Decode-sized T at shapes on either side of the decode kernel's limits:
    K not a multiple of 64, N not a multiple of 8, dense outlier sets, tiny
    shapes."""
    w = inputs.random_small(T, K, N, ncols, seed=T * 5 + K + N, tau=tau)
    run_and_compare(orc, w.X, w.W, tau, what=f"decode shape T{T} K{K} N{N} tau{tau}")
