"""Per-row FP8 (E4M3) quantisation and the GEMM over the codes, on the GPU.

RedFuser page, sections 1 and 4: FP8 quantisation followed by GEMM is a cascade
of reductions. The quantised codes decide integers, so both sides take them in
float32 (x * (448 / amax)) and they must match the oracle's bit for bit, as
must the scales. The GEMM accumulates products of E4M3 values (each exact in
float32) on the tensor cores and rounds C to bf16: the bound below allows half
a bf16 ulp of |C| plus 2^-13 of the sum of |products| (an accumulator holding
at least 13 significant bits).
"""

import numpy as np
import pytest
import torch

import oracle
from online_softmax_attention_rf_gb300 import api, inputs
from tests.helpers import f64

pytestmark = pytest.mark.gpu


def _decode(codes):
    return codes.cpu().view(torch.float8_e4m3fn).to(torch.float64).numpy()


@pytest.mark.parametrize("rows,K", [(7, 16), (33, 128), (5, 4096), (3, 32768), (4, 1040)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_rowquant_matches_oracle_bit_for_bit(cuda_device, rows, K, dtype):
    if dtype == "f32" and K * 4 > 64 * 1024:
        K //= 2
    g = torch.Generator().manual_seed(rows * 100 + K)
    x = torch.randn(rows, K, generator=g) * torch.logspace(-3, 3, rows)[:, None]
    x[0, :] = 0.0                                     # an all-zero row
    if rows > 2:
        x[1, 5] = 3000.0                              # most of the row falls to subnormal codes
    x = x.to(inputs.TORCH_DTYPES[dtype])
    q, sc = api.rowquant_e4m3(x.cuda())
    assert api.device_status() == 0
    rq, rsc = oracle.rowquant_e4m3(f64(x))
    assert np.array_equal(_decode(q), rq)
    assert np.array_equal(sc.cpu().numpy(), rsc)
    assert np.array_equal(q.cpu().numpy(), oracle.e4m3_code(rq))


def _check_gemm(c, qa, sa, qw, sw):
    ref = oracle.fp8_gemm(qa, sa, qw, sw)
    mag = np.outer(np.asarray(sa, np.float64), np.asarray(sw, np.float64)) * \
        (np.abs(qa) @ np.abs(qw).T)
    tol = 2.0 ** -8 * np.abs(ref) + 2.0 ** -13 * mag + 1e-30
    err = np.abs(f64(c) - ref)
    assert (err <= tol).all(), "C: worst err/tol %.3g" % (err / tol).max()
    return float((err / np.maximum(mag, 1e-30)).max())


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (256, 512, 1024), (384, 256, 640)])
def test_fp8_gemm_matches_oracle(cuda_device, M, N, K):
    a, w = inputs.make_gemm_operands(M, N, K, M + N + K)
    qa, sa = oracle.rowquant_e4m3(f64(a))
    qw, sw = oracle.rowquant_e4m3(f64(w))
    ca = torch.from_numpy(oracle.e4m3_code(qa)).cuda()
    cw = torch.from_numpy(oracle.e4m3_code(qw)).cuda()
    c = api.fp8_gemm(ca, torch.from_numpy(sa).cuda(), cw, torch.from_numpy(sw).cuda())
    assert api.device_status() == 0
    _check_gemm(c, qa, sa, qw, sw)


def test_quantise_then_gemm_chain(cuda_device):
    """The whole cascade on the GPU (quantise A, quantise W, GEMM) against
    the oracle's chain on the same bf16 inputs."""
    M, N, K = 256, 512, 2048
    a, w = inputs.make_gemm_operands(M, N, K, 5)
    qa_d, sa_d = api.rowquant_e4m3(a.cuda())
    qw_d, sw_d = api.rowquant_e4m3(w.cuda())
    c = api.fp8_gemm(qa_d, sa_d, qw_d, sw_d)
    assert api.device_status() == 0
    qa, sa = oracle.rowquant_e4m3(f64(a))
    qw, sw = oracle.rowquant_e4m3(f64(w))
    assert np.array_equal(_decode(qa_d), qa) and np.array_equal(_decode(qw_d), qw)
    _check_gemm(c, qa, sa, qw, sw)
    # and the quantised product is close to the bf16 product
    exact = f64(a) @ f64(w).T
    assert np.abs(f64(c) - exact).max() <= 0.1 * np.abs(exact).max()


def test_fp8_full_size_sampled(cuda_device):
    """The 8192^3 workload in the launch configuration the benchmark times;
    16 x 16 sampled outputs against the oracle."""
    wk = inputs.CASCADE_WORKLOADS["fp8_gemm"]
    a, w = inputs.make_gemm_operands(wk["M"], wk["N"], wk["K"], wk["seed"])
    qa_d, sa_d = api.rowquant_e4m3(a.cuda())
    qw_d, sw_d = api.rowquant_e4m3(w.cuda())
    c = api.fp8_gemm(qa_d, sa_d, qw_d, sw_d)
    assert api.device_status() == 0
    rng = np.random.default_rng(3)
    rows = np.sort(rng.choice(wk["M"], 16, replace=False))
    cols = np.sort(rng.choice(wk["N"], 16, replace=False))
    qa, sa = oracle.rowquant_e4m3(f64(a[rows]))
    qw, sw = oracle.rowquant_e4m3(f64(w[cols]))
    assert np.array_equal(_decode(qa_d[rows]), qa) and np.array_equal(_decode(qw_d[cols]), qw)
    _check_gemm(c[rows][:, cols], qa, sa, qw, sw)
