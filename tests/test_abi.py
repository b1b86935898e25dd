"""The C-ABI library builds for sm_103a, loads, exports every symbol the
header declares, and rejects bad arguments on the host before touching the
GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gbce.h")


@pytest.fixture(scope="module")
def lib():
    from softmax_cross_entropy_gb300 import build, _lib
    build.build()
    return _lib.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ce_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("ce_fwd", "ce_bwd", "ce_device_status", "ce_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_covers_every_declared_symbol():
    from softmax_cross_entropy_gb300 import _lib
    assert sorted(_lib.SIGNATURES) == declared_functions()


def test_library_targets_sm_103a():
    from softmax_cross_entropy_gb300 import build
    assert "arch=compute_103a,code=sm_103a" in " ".join(build.ARCH)


def test_status_strings(lib):
    from softmax_cross_entropy_gb300 import _lib
    for code in range(6):
        assert _lib.ce_status_string(code)
    assert _lib.ce_status_string(99) == "unknown status"


def _fwd(lib, **over):
    from softmax_cross_entropy_gb300 import _lib
    a = dict(logits=16, dtype=_lib.CE_BF16, rows=4, V=8, target=32, weight=None,
             ignore_index=-100, label_smoothing=0.0, lse_square_scale=0.0, softcap=0.0,
             reduction=_lib.CE_RED_MEAN, flags=0, loss=48, z_loss=None, acc=None, pred=None,
             stream=None)
    a.update(over)
    return _lib.ce_fwd(**a)


@pytest.mark.parametrize("over", [
    dict(dtype=7), dict(rows=-1), dict(V=0), dict(V=-5), dict(reduction=3),
    dict(label_smoothing=-0.1), dict(label_smoothing=1.5), dict(label_smoothing=float("nan")),
    dict(lse_square_scale=float("inf")), dict(softcap=-1.0), dict(softcap=float("nan")),
    dict(softcap=float("inf")), dict(loss=None), dict(logits=None), dict(target=None),
    dict(flags=2), dict(flags=4), dict(flags=8), dict(flags=64),
])
def test_invalid_arguments_are_rejected_on_the_host(lib, over):
    from softmax_cross_entropy_gb300 import _lib
    assert _fwd(lib, **over) == _lib.CE_ERR_INVALID_ARG


def test_oversized_vocabulary_is_unsupported(lib):
    from softmax_cross_entropy_gb300 import _lib
    assert _fwd(lib, V=2**31) == _lib.CE_ERR_UNSUPPORTED


def test_empty_batch_with_no_reduction_is_a_no_op(lib):
    from softmax_cross_entropy_gb300 import _lib
    assert _fwd(lib, rows=0, logits=None, target=None, reduction=_lib.CE_RED_NONE) == _lib.CE_OK


@pytest.mark.parametrize("over", [dict(dtype=5), dict(rows=-2), dict(V=0),
                                  dict(grad_output=None), dict(dlogits=None)])
def test_bwd_invalid_arguments(lib, over):
    from softmax_cross_entropy_gb300 import _lib
    a = dict(grad_output=16, grad_per_row=0, dlogits=32, dtype=_lib.CE_F32, rows=3, V=5,
             stream=None)
    a.update(over)
    assert _lib.ce_bwd(**a) == _lib.CE_ERR_INVALID_ARG


def test_fp16_dtype_is_part_of_the_boundary(lib):
    from softmax_cross_entropy_gb300 import _lib
    assert _lib.CE_F16 == 2
    # an fp16 call with an invalid argument fails on the argument, not on the dtype
    assert _fwd(lib, dtype=_lib.CE_F16, rows=-1) == _lib.CE_ERR_INVALID_ARG
    assert _fwd(lib, dtype=3) == _lib.CE_ERR_INVALID_ARG


def _shard(lib, **over):
    from softmax_cross_entropy_gb300 import _lib
    a = dict(logits=16, dtype=_lib.CE_BF16, rows=4, V=8, target=32, weight=None,
             ignore_index=-100, label_smoothing=0.0, lse_square_scale=0.0, softcap=0.0,
             reduction=_lib.CE_RED_MEAN, flags=0, loss=48, z_loss=None, acc=None, pred=None,
             batch_counts=64, stream=None)
    a.update(over)
    return _lib.ce_fwd_shard(**a)


@pytest.mark.parametrize("over", [dict(batch_counts=None), dict(dtype=9), dict(rows=-1),
                                  dict(loss=None), dict(flags=64), dict(softcap=-2.0)])
def test_shard_invalid_arguments(lib, over):
    from softmax_cross_entropy_gb300 import _lib
    assert _shard(lib, **over) == _lib.CE_ERR_INVALID_ARG


@pytest.mark.parametrize("over", [dict(counts=None), dict(rows=-1), dict(V=0),
                                  dict(flags=1), dict(flags=32), dict(target=None)])
def test_count_invalid_arguments(lib, over):
    from softmax_cross_entropy_gb300 import _lib
    a = dict(target=16, weight=None, rows=5, V=10, ignore_index=-100, flags=0, counts=32,
             stream=None)
    a.update(over)
    assert _lib.ce_count(**a) == _lib.CE_ERR_INVALID_ARG


def test_python_api_rejects_rank_1_and_nd_logits():
    torch = pytest.importorskip("torch")
    import softmax_cross_entropy_gb300 as ce
    t = torch.zeros(4, dtype=torch.int64)
    with pytest.raises(ValueError):
        ce.cross_entropy(torch.zeros(4), t)          # rank 1
    with pytest.raises(ValueError):
        ce.cross_entropy(torch.zeros(2, 4, 5), t)    # N-D logits on the CPU
    with pytest.raises(ValueError):
        ce.cross_entropy(torch.zeros(4, 5), t)       # not on a CUDA device


def test_nvtx_ranges_only_when_asked(monkeypatch):
    # the wrapper's NVTX ranges push and pop in pairs when enabled, and call
    # nothing when not
    import torch
    import softmax_cross_entropy_gb300 as gbce
    calls = []
    monkeypatch.setattr(torch.cuda.nvtx, "range_push", lambda n: calls.append(("push", n)))
    monkeypatch.setattr(torch.cuda.nvtx, "range_pop", lambda: calls.append(("pop",)))
    monkeypatch.setattr(gbce, "_NVTX", False)
    with gbce._Range("gbce.x"):
        pass
    assert calls == []
    monkeypatch.setattr(gbce, "_NVTX", True)
    try:
        with gbce._Range("gbce.y"):
            raise KeyError("inside")
    except KeyError:
        pass
    assert calls == [("push", "gbce.y"), ("pop",)]


def test_bench_provenance_names_the_sources():
    # the bench line records what produced it: the headline kernel's source
    # hash always, the git commit when the tree is a checkout
    import bench
    p = bench.provenance()
    assert p["headline_kernel_sources"] == bench.kernel_source_hash()
    assert len(p["headline_kernel_sources"]) == 16
    assert p["git_sha"] is None or len(p["git_sha"]) == 40
