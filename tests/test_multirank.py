"""Multi-rank logic on CPU with two gloo ranks (no GPU).

* The benchmark's plumbing: barrier and max-over-ranks timing.
* Splitting the output channels across ranks needs no exchange: every rank
  computes the same outlier set from the replicated X, and the concatenated
  slices equal the single-device result bit for bit.
* Splitting the tokens across ranks needs exactly one exchange to match the
  single-device result: an OR all-reduce of the K-column outlier mask between
  the column scan and the quantization of the rows; without it the ranks'
  outlier sets (and so their results) differ.
"""

import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import inputs

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, q):
    import torch
    import torch.distributed as dist
    try:
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dist.init_process_group("gloo", rank=rank, world_size=WORLD)
        import bench
        import oracle
        orc = oracle.get()
        out = {}

        # bench plumbing: barrier + max over ranks
        bench.barrier(WORLD)
        out["max"] = bench.max_over_ranks(float(rank + 1) * 1.5, WORLD)

        w = inputs.random_small(12, 96, 40, 3, seed=21)
        w.X = w.X.copy()
        w.X[8, 5] = 9.0  # an outlier seen only by the rank holding row 8
        Wq, sw = orc.quantize_weight(w.W)
        full = orc.linear(w.X, Wq, sw, w.W, w.tau)

        # output-channel split: no exchange
        n0, n1 = rank * 20, (rank + 1) * 20
        mine = orc.linear(w.X, Wq[n0:n1], sw[n0:n1], w.W[n0:n1], w.tau)
        # fp16 bit patterns travel as int32 (gloo has no 16-bit integer type)
        ys = [torch.zeros(12, 20, dtype=torch.int32) for _ in range(WORLD)]
        dist.all_gather(ys, torch.from_numpy(mine["Y"].view(np.uint16).astype(np.int32)))
        y_cat = torch.cat(ys, dim=1).numpy().astype(np.uint16)
        out["nsplit_equal"] = bool(np.array_equal(y_cat, full["Y"].view(np.uint16)))

        # the same split for the other forms of the layer: a bias (split with
        # the channels), only the int8 weight, and bf16 X / W / bias / Y
        bias = inputs.bias(40, 96, seed=5)
        Wb = torch.from_numpy(w.W.astype(np.float32)).to(torch.bfloat16)
        Wb = Wb.view(torch.int16).numpy().view(np.uint16)
        Xb = torch.from_numpy(w.X.astype(np.float32)).to(torch.bfloat16)
        Xb = Xb.view(torch.int16).numpy().view(np.uint16)
        bb = torch.from_numpy(bias.astype(np.float32)).to(torch.bfloat16)
        bb = bb.view(torch.int16).numpy().view(np.uint16)
        Wqb, swb = orc.quantize_weight(Wb, fmt="bf16")
        forms = {
            "bias": (dict(X16=w.X, Wq=Wq, sw=sw, W16=w.W, bias=bias), {}),
            "wq_only": (dict(X16=w.X, Wq=Wq, sw=sw, W16=None, bias=bias), {}),
            "bf16": (dict(X16=Xb, Wq=Wqb, sw=swb, W16=Wb, bias=bb), {"fmt": "bf16"}),
        }
        for name, (a, kw) in forms.items():
            full_f = orc.linear(a["X16"], a["Wq"], a["sw"], a["W16"], w.tau, bias=a["bias"], **kw)
            mine_f = orc.linear(a["X16"], a["Wq"][n0:n1], a["sw"][n0:n1],
                                None if a["W16"] is None else a["W16"][n0:n1], w.tau,
                                bias=a["bias"][n0:n1], **kw)
            ys = [torch.zeros(12, 20, dtype=torch.int32) for _ in range(WORLD)]
            dist.all_gather(ys, torch.from_numpy(mine_f["Y"].view(np.uint16).astype(np.int32)))
            y_cat = torch.cat(ys, dim=1).numpy().astype(np.uint16)
            out["nsplit_equal_" + name] = bool(np.array_equal(y_cat, full_f["Y"].view(np.uint16)))

        # token split: OR all-reduce of the outlier column mask
        t0, t1 = rank * 6, (rank + 1) * 6
        X_loc = w.X[t0:t1]
        O_loc = orc.outlier_columns(X_loc, w.tau)
        mask = torch.zeros(w.K, dtype=torch.int32)
        mask[torch.from_numpy(O_loc.astype(np.int64))] = 1
        dist.all_reduce(mask, op=dist.ReduceOp.MAX)  # logical OR of 0/1 flags
        O_glob = np.flatnonzero(mask.numpy()).astype(np.int32)
        out["mask_equals_full_scan"] = bool(np.array_equal(O_glob, full["O"]))
        Xq, sx, XO = orc.quantize_activations(X_loc, O_glob)
        acc = orc.int8_matmul(Xq, Wq)
        out["tsplit_codes_equal"] = bool(np.array_equal(Xq, full["Xq"][t0:t1]))
        out["tsplit_acc_equal"] = bool(np.array_equal(acc, full["acc"][t0:t1]))
        # without the exchange the local outlier set differs on some rank
        out["local_differs"] = not np.array_equal(O_loc, full["O"])
        q.put((rank, out))
        dist.destroy_process_group()
    except Exception as e:  # report to the parent instead of hanging it
        q.put((rank, {"error": repr(e)}))


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    res = {}
    try:
        for _ in range(WORLD):
            r, out = q.get(timeout=240)
            res[r] = out
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.kill()
    for r in range(WORLD):
        assert "error" not in res[r], res[r]
        assert res[r]["max"] == pytest.approx(3.0)
        assert res[r]["nsplit_equal"]
        for name in ("bias", "wq_only", "bf16"):
            assert res[r]["nsplit_equal_" + name], name
        assert res[r]["mask_equals_full_scan"]
        assert res[r]["tsplit_codes_equal"] and res[r]["tsplit_acc_equal"]
    # rank 0 does not see column 5's outlier: without the exchange it differs
    assert res[0]["local_differs"]
