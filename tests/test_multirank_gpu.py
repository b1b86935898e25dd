"""The row-sharded mean on the device path, across two processes: each rank
counts its rows on the GPU (ce_count), the two counts are all-reduced over
`gloo` (through host memory), and each rank runs the public cross_entropy
with those batch counts (ce_fwd_shard). The ranks' loss outputs must add up
to the oracle's whole-batch mean, and every rank's gradient rows must be the
oracle's rows of the whole-batch gradient.

Both ranks share the one GPU of the test machine. Their kernels never wait
on each other: the only exchange is the host-side all-reduce between the
count and the forward."""
import os
import socket

import numpy as np
import pytest

import workloads

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case(spec):
    return workloads.random_case(*spec["args"], **spec["kw"])


def _rank_main(rank, world, port, spec, out_dir):
    import torch
    import torch.distributed as dist

    import softmax_cross_entropy_gb300 as ce
    from softmax_cross_entropy_gb300 import distributed as cedist
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        case = _case(spec)
        lo, hi = cedist.shard_rows(case.rows, rank, world)
        dt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[case.dtype]
        xs = case.x[lo:hi]
        if case.dtype == "f32":
            x = torch.from_numpy(np.ascontiguousarray(xs))
        else:
            x = torch.from_numpy(np.ascontiguousarray(xs).view(np.int16)).view(dt)
        x = x.cuda().requires_grad_()
        t = torch.from_numpy(np.ascontiguousarray(case.target[lo:hi])).cuda()
        w = None if case.weight is None else torch.from_numpy(case.weight).cuda()
        counts = cedist.batch_counts(t, case.V, w, case.ignore_index)
        out = ce.cross_entropy(x, t, weight=w, ignore_index=case.ignore_index,
                               lse_square_scale=case.lse_square_scale,
                               label_smoothing=case.label_smoothing, softcap=case.softcap,
                               return_z_loss=True, return_token_accuracy=True,
                               batch_counts=counts)
        out.loss.backward()
        torch.cuda.synchronize()
        grad = x.grad.float().cpu().numpy().astype(np.float64)
        np.save(os.path.join(out_dir, f"grad{rank}.npy"), grad)
        np.save(os.path.join(out_dir, f"scal{rank}.npy"),
                np.array([out.loss.item(), out.z_loss.item(), out.token_accuracy.item(),
                          counts[0].item(), counts[1].item(), lo, hi]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("spec", [
    {"args": (41, 301, 8192), "kw": dict(dtype="bf16")},
    {"args": (42, 97, 4096), "kw": dict(dtype="f32", weight=True, label_smoothing=0.1,
                                        lse_square_scale=1e-3)},
    {"args": (43, 64, 32000), "kw": dict(dtype="bf16", softcap=20.0, label_smoothing=0.05)},
    {"args": (44, 40, 65536), "kw": dict(dtype="bf16", ignore_frac=1.0)},  # all ignored
], ids=["bf16-8192", "f32-weighted", "bf16-softcap", "all-ignored"])
def test_two_process_sharded_mean_matches_whole_batch(tmp_path, spec):
    import math
    import multiprocessing as mp

    import oracle
    from ce_gpu import assert_grad_close, assert_loss_close
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from softmax_cross_entropy_gb300 import build
    build.build()  # once, before the ranks load it
    world = 2
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, spec, str(tmp_path)))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0, f"rank exited with {p.exitcode}"
    case = _case(spec)
    ref = oracle.forward(case.x, case.target, dtype=case.dtype, weight=case.weight,
                         **case.options())
    scal = [np.load(tmp_path / f"scal{r}.npy") for r in range(world)]
    loss = sum(float(s[0]) for s in scal)
    zl = sum(float(s[1]) for s in scal)
    for s in scal:  # every rank saw the batch counts
        assert s[4] == np.sum(case.target != case.ignore_index)
    if math.isnan(ref["loss"]):
        assert all(math.isnan(float(s[0])) for s in scal)
    else:
        assert_loss_close(loss, ref["loss"], case.dtype)
        assert_loss_close(zl, ref["z_loss"], case.dtype, "z_loss")
        acc = sum(float(s[2]) for s in scal)
        assert np.float32(acc) == np.float32(ref["acc"]) or abs(acc - ref["acc"]) < 1e-6
    grad = np.concatenate([np.load(tmp_path / f"grad{r}.npy") for r in range(world)])
    assert_grad_close(grad, ref["grad"], case.dtype)
