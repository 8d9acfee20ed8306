"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and the oracle on the same seeded inputs, and compare.

Bit-exact: outlier list and count, activation codes, row scales, weight codes
and scales, int32 accumulators.  Y (fp16) within the tolerance of the layer:
for every row t, max_n |Y - Y_ref| <= 2e-3 * max_n |Y_ref|, and over the whole
compared block ||Y - Y_ref||_F <= 1e-3 ||Y_ref||_F.  Infinite reference
values (integer inputs whose products exceed fp16's range) must be matched by
infinities of the same sign.
"""

from __future__ import annotations

import numpy as np

ROW_TOL = 2e-3
FRO_TOL = 1e-3


def check_y(y_gpu: np.ndarray, y_ref: np.ndarray, what: str = ""):
    g = y_gpu.astype(np.float64)
    r = y_ref.astype(np.float64)
    inf_ref = np.isinf(r)
    assert np.array_equal(np.isinf(g), inf_ref), f"{what}: infinities differ"
    assert np.array_equal(np.sign(g[inf_ref]), np.sign(r[inf_ref])), f"{what}: inf signs"
    assert not np.isnan(g).any(), f"{what}: NaN in Y"
    fin = ~inf_ref
    rz = np.where(fin, r, 0.0)
    err = np.abs(np.where(fin, g - r, 0.0))
    row_max = np.abs(rz).max(axis=1)
    row_err = err.max(axis=1)
    bad = np.flatnonzero(row_err > ROW_TOL * row_max)
    assert len(bad) == 0, (f"{what}: row tolerance, rows {bad[:5]}, err {row_err[bad[:5]]}, "
                           f"rowmax {row_max[bad[:5]]}")
    den = np.sqrt((rz ** 2).sum())
    if den > 0:
        rel = np.sqrt((err ** 2).sum()) / den
        assert rel <= FRO_TOL, f"{what}: relative Frobenius error {rel}"
    else:
        assert err.max(initial=0.0) == 0.0


def sample_rows(T: int, n: int = 64, seed: int = 0) -> np.ndarray:
    """Seeded sample of rows plus rows 0 and T-1, ascending, unique."""
    rng = np.random.default_rng(seed + 1000)
    rows = set(rng.choice(T, size=min(n, T), replace=False).tolist()) | {0, T - 1}
    return np.array(sorted(rows), dtype=np.int64)


def run_and_compare(orc, X16: np.ndarray, W16: np.ndarray, tau: float, rows=None,
                    what: str = "", check_weights: bool = True, opts: int = 0):
    """CUDA path (debug entry point, same kernels as bnb_int8_linear; with
    ``opts``, bnb_int8_linear_opts with those per-call options) vs oracle."""
    import torch

    from int8_mixed_precision_04_b300 import binding

    T, K = X16.shape
    N = W16.shape[0]
    X = torch.from_numpy(np.ascontiguousarray(X16)).cuda()
    W = torch.from_numpy(np.ascontiguousarray(W16)).cuda()
    Wq, sw = binding.quantize_weight(W)
    r = (binding.linear_opts(X, Wq, sw, W, tau, opts, debug=True) if opts
         else binding.linear_debug(X, Wq, sw, W, tau))
    torch.cuda.synchronize()
    assert binding.last_device_status(r["workspace"]) == 0
    Wq_o, sw_o = orc.quantize_weight(W16)
    if check_weights:
        assert np.array_equal(Wq.cpu().numpy(), Wq_o), f"{what}: weight codes"
        assert np.array_equal(sw.cpu().numpy(), sw_o), f"{what}: weight scales"
    ref = orc.linear(X16, Wq_o, sw_o, W16, tau, rows=rows)
    nO = int(r["nO"].item())
    O = r["O"][:nO].cpu().numpy()
    assert np.array_equal(O, ref["O"]), f"{what}: outlier list {O[:8]} vs {ref['O'][:8]}"
    assert np.array_equal(r["sx"].cpu().numpy(), ref["sx"]), f"{what}: row scales"
    xq = r["Xq"].cpu().numpy()
    if not np.array_equal(xq, ref["Xq"]):
        bad = np.argwhere(xq != ref["Xq"])[:5]
        raise AssertionError(f"{what}: activation codes differ at {bad.tolist()}")
    rows_t = torch.from_numpy(ref["rows"]).cuda()
    acc = r["acc"].index_select(0, rows_t).cpu().numpy()
    if not np.array_equal(acc, ref["acc"]):
        bad = np.argwhere(acc != ref["acc"])[:5]
        raise AssertionError(f"{what}: int32 accumulators differ at {bad.tolist()}: "
                             f"{acc[tuple(bad[0])]} vs {ref['acc'][tuple(bad[0])]}")
    y = r["Y"].index_select(0, rows_t).cpu().numpy()
    check_y(y, ref["Y"], what)
    return r, ref
