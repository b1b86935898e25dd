"""GPU parity of the tensor-core GEMM of the fused linear cross-entropy
(ce_gemm_abt: C = A @ B^T + bias on tcgen05, operands staged by TMA) against
the oracle's float64 logits (oracle.linear) on seeded inputs. C is an fp32
sum of exact bf16 / fp16 products, so each entry is within
K * 2^-23 * sum_k |a_ik b_jk| of the exact value (fp32 accumulation,
rounding or truncation in the adds), plus one fp32 rounding of the bias
sum."""
import math

import numpy as np
import pytest

import workloads

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
CE_DT = {"bf16": 1, "f16": 2}


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from softmax_cross_entropy_gb300 import build, _lib
    build.build()
    _lib.load()


def dev16(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
        torch.bfloat16 if dtype == "bf16" else torch.float16).cuda()


def run(M, N, K, dtype, with_bias, seed):
    import oracle
    from softmax_cross_entropy_gb300 import _lib
    a = workloads.random_case(seed, M, K, dtype=dtype, std=1.0, ignore_frac=0.0).x
    b = workloads.random_case(seed + 1, N, K, dtype=dtype, std=1.0 / math.sqrt(K),
                              ignore_frac=0.0).x
    bias = np.random.default_rng(seed).normal(0, 1, N).astype(np.float32) if with_bias else None
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    db = None if bias is None else torch.from_numpy(bias).cuda()
    st = torch.cuda.current_stream().cuda_stream
    da, dbm = dev16(a, dtype), dev16(b, dtype)  # held until the kernel has run
    rc = _lib.ce_gemm_abt(da.data_ptr(), dbm.data_ptr(), CE_DT[dtype], M, N, K, C.data_ptr(),
                          None if db is None else db.data_ptr(), st)
    assert rc == _lib.CE_OK, (_lib.ce_status_string(rc), _lib.ce_last_error())
    assert _lib.ce_device_status(st) == 0
    got = C.double().cpu().numpy()
    want = oracle.linear(a, b, dtype=dtype, bias=bias)
    bound = K * 2.0 ** -23 * (np.abs(oracle.decode(a, dtype)) @ np.abs(oracle.decode(b, dtype)).T)
    bound += 2.0 ** -23 * np.abs(want) + 1e-30
    err = np.abs(got - want)
    assert np.all(np.isfinite(got))
    bad = err > bound
    assert not bad.any(), (f"{bad.sum()} of {bad.size} out of bound; first at "
                           f"{tuple(np.argwhere(bad)[0])}: got {got[bad][0]} want {want[bad][0]}")


def test_one_tile():
    run(128, 256, 64, "bf16", False, 1)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (300, 1000, 136), (1, 17, 8), (129, 257, 520),
                                   (1046, 2048, 1024)])
@pytest.mark.parametrize("with_bias", [False, True])
def test_gemm_parity(dtype, M, N, K, with_bias):
    run(M, N, K, dtype, with_bias, M + N + K)


def test_unsupported_k():
    from softmax_cross_entropy_gb300 import _lib
    a = torch.zeros(4, 12, dtype=torch.bfloat16, device="cuda")
    C = torch.empty(4, 4, device="cuda")
    rc = _lib.ce_gemm_abt(a.data_ptr(), a.data_ptr(), 1, 4, 4, 12, C.data_ptr(), None,
                          torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.CE_ERR_UNSUPPORTED


def _stored(x, dtype, transpose):
    """The device copy of a 16-bit operand given as [rows, cols] bits,
    stored as is or transposed (MN-major storage)."""
    return dev16(np.ascontiguousarray(x.T) if transpose else x, dtype)


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("c_mode", [0, 1, 2])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 520, 136), (8, 24, 8),
                                   (1048, 2056, 1032)])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("bm", ["128", "256"])
def test_gemm_layouts_and_outputs(monkeypatch, a_mn, b_mn, c_mode, M, N, K, dtype, bm):
    # ce_gemm: A [M, K] and B [K, N] stored K-major or MN-major; C written
    # in fp32, added to in fp32, or rounded to the operand type; tiles of
    # 128 or 256 rows (GBCE_TC_BM). The reference is the oracle's float64
    # product of the same bits.
    import oracle
    from softmax_cross_entropy_gb300 import _lib
    monkeypatch.setenv("GBCE_TC_BM", bm)
    seed = 7 * M + 3 * N + K + 11 * a_mn + 13 * b_mn + 17 * c_mode
    a = workloads.random_case(seed, M, K, dtype=dtype, std=1.0, ignore_frac=0.0).x   # [M, K]
    bt = workloads.random_case(seed + 1, N, K, dtype=dtype, std=1.0 / math.sqrt(K),
                               ignore_frac=0.0).x                                    # [N, K] = B^T
    da = _stored(a, dtype, a_mn)
    # (B K-major is stored as [N, K] = bt; MN-major as [K, N] = bt^T)
    if b_mn:
        db = dev16(np.ascontiguousarray(bt.T), dtype)
    else:
        db = dev16(bt, dtype)
    rng = np.random.default_rng(seed)
    c0 = rng.normal(0, 1, (M, N)).astype(np.float32)
    if c_mode == 2:
        C = torch.full((M, N), float("nan"), device="cuda").to(
            torch.bfloat16 if dtype == "bf16" else torch.float16)
    elif c_mode == 1:
        C = torch.from_numpy(c0).cuda()
    else:
        C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    rc = _lib.ce_gemm(da.data_ptr(), a_mn, db.data_ptr(), b_mn, CE_DT[dtype], M, N, K,
                      C.data_ptr(), c_mode, None, st)
    assert rc == _lib.CE_OK, (_lib.ce_status_string(rc), _lib.ce_last_error())
    assert _lib.ce_device_status(st) == 0
    got = C.double().cpu().numpy()
    want = oracle.linear(a, bt, dtype=dtype)
    bound = K * 2.0 ** -23 * (np.abs(oracle.decode(a, dtype)) @ np.abs(oracle.decode(bt, dtype)).T)
    if c_mode == 1:
        want = want + c0.astype(np.float64)
    bound += 2.0 ** -23 * np.abs(want) + 1e-30
    if c_mode == 2:  # one rounding to the 16-bit type
        bound += np.abs(want) * (2.0 ** -8 if dtype == "bf16" else 2.0 ** -11) + 2.0 ** -24
    err = np.abs(got - want)
    assert np.all(np.isfinite(got))
    bad = err > bound
    assert not bad.any(), (f"{bad.sum()} of {bad.size} out of bound; first at "
                           f"{tuple(np.argwhere(bad)[0])}: got {got[bad][0]} want {want[bad][0]}")


@pytest.mark.parametrize("bm", ["128", "256"])
@pytest.mark.parametrize("c_mode", [0, 1, 2])
@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (1, 1)])
def test_gemm_many_rounds(monkeypatch, bm, c_mode, a_mn, b_mn):
    # 2048 x 8192 with a ragged K: 256 or 512 tiles, so each persistent CTA
    # runs two to four tiles and the stage ring and the accumulator
    # barriers wrap their phases several times
    test_gemm_layouts_and_outputs(monkeypatch, a_mn, b_mn, c_mode, 2048, 8192, 72, "bf16", bm)


def test_gemm_rejects_bad_operands():
    from softmax_cross_entropy_gb300 import _lib
    a = torch.zeros(16, 12, dtype=torch.bfloat16, device="cuda")
    C = torch.empty(16, 16, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    # an MN-major A whose M (12 per row of storage) is not a multiple of 8
    assert _lib.ce_gemm(a.data_ptr(), 1, a.data_ptr(), 0, 1, 12, 16, 16, C.data_ptr(), 0, None,
                        st) == _lib.CE_ERR_UNSUPPORTED
    # a bias with an accumulating output
    b = torch.zeros(16, dtype=torch.float32, device="cuda")
    assert _lib.ce_gemm(a.data_ptr(), 0, a.data_ptr(), 0, 1, 16, 16, 8, C.data_ptr(), 1,
                        b.data_ptr(), st) == _lib.CE_ERR_INVALID_ARG
