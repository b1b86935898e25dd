"""Row-sharded mean across ranks, on CPU `gloo` ranks (world size 2): the
shard statistics combined by softmax_cross_entropy_gb300.distributed must
give the unsharded oracle's mean loss, accuracy and gradient."""
import os
import socket

import numpy as np
import pytest

import workloads

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, case_args, out_dir):
    import torch.distributed as dist

    import oracle
    from softmax_cross_entropy_gb300 import distributed as cedist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        case = workloads.random_case(*case_args["args"], **case_args["kw"])
        lo, hi = cedist.shard_rows(case.rows, rank, world)
        x, t = case.x[lo:hi], case.target[lo:hi]
        opts = case.options()
        opts["reduction"] = "sum"
        s = oracle.forward(x, t, dtype=case.dtype, weight=case.weight, want_grad=False, **opts)
        opts["reduction"] = "mean"
        m = oracle.forward(x, t, dtype=case.dtype, weight=case.weight, **opts)
        D_loc, n_loc = cedist.local_denominator(t, case.ignore_index, case.weight, case.V)
        n_correct = float(np.nansum(s["acc"]) * n_loc) if n_loc else 0.0
        g = cedist.reduce_mean(float(s["loss"]), float(s["z_loss"]), n_correct, D_loc, n_loc)
        grad = oracle.backward(m["grad"], cedist.mean_grad_factor(D_loc, g["D"]))
        np.save(os.path.join(out_dir, f"grad{rank}.npy"), grad)
        np.save(os.path.join(out_dir, f"scal{rank}.npy"),
                np.array([g["loss"], g["z_loss"], g["acc"], lo, hi]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("kw", [
    dict(label_smoothing=0.1, lse_square_scale=1e-3),
    dict(weight=True, label_smoothing=0.05),
    dict(ignore_frac=1.0),  # every row ignored: NaN mean, zero gradients
])
def test_sharded_mean_matches_unsharded_oracle(tmp_path, kw):
    import multiprocessing as mp

    import oracle
    world = 2
    case_args = {"args": (3, 37, 96), "kw": dict(dtype="f32", **kw)}
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, case_args, str(tmp_path)))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    case = workloads.random_case(*case_args["args"], **case_args["kw"])
    ref = oracle.forward(case.x, case.target, dtype="f32", weight=case.weight, **case.options())
    acc_ref = oracle.forward(case.x, case.target, dtype="f32", weight=case.weight,
                             want_grad=False, **{**case.options(), "reduction": "sum"})["acc"]
    grads = []
    for r in range(world):
        sc = np.load(tmp_path / f"scal{r}.npy")
        for got, want in ((sc[0], ref["loss"]), (sc[1], ref["z_loss"]), (sc[2], acc_ref)):
            if np.isnan(want):
                assert np.isnan(got)
            else:
                assert got == pytest.approx(want, rel=1e-12)
        grads.append(np.load(tmp_path / f"grad{r}.npy"))
    np.testing.assert_allclose(np.concatenate(grads), ref["grad"], rtol=1e-12, atol=1e-300)


def test_shard_rows_partition():
    from softmax_cross_entropy_gb300.distributed import shard_rows
    for rows in (0, 1, 7, 4096, 1023):
        for world in (1, 2, 3, 8):
            parts = [shard_rows(rows, r, world) for r in range(world)]
            assert parts[0][0] == 0 and parts[-1][1] == rows
            assert all(a[1] == b[0] for a, b in zip(parts, parts[1:]))
            sizes = [b - a for a, b in parts]
            assert max(sizes) - min(sizes) <= 1
