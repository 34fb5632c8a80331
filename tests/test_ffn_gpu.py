"""The BitNet FFN pieces around the BitLinear, against the oracle: the
sub-layer RMS norm followed by the activation quantisation (reading R9: the
exact mean of squares, so x_q and s are bit-exact) and the squared-ReLU
epilogue (reading R10), on every kernel path."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

Y_RTOL = 1e-5


@pytest.fixture(scope="module")
def bl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from ternary_weight_06_b300 import build

    build.build()
    import ternary_weight_06_b300 as mod

    return mod


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("K", [1, 63, 2560, 6912, 40000])
@pytest.mark.parametrize("with_gain", [False, True])
def test_rmsnorm_quant_act(bl, dtype, K, with_gain):
    g = torch.Generator().manual_seed(K + with_gain)
    X = torch.randn((7, K), generator=g) * 3.0
    X[1] = 0.0  # an all-zero token
    X[2] *= 1e4
    X[3] *= 1e30  # squares overflow fp32 unless scaled
    X[4] *= 1e-40  # subnormal in fp32 (and bf16)
    X = X.to(dtype)
    gain = (torch.rand((K,), generator=g) * 2.0).to(torch.float32) if with_gain else None
    xq_ref, s_ref = oracle.rmsnorm_quant_act(X.to(torch.float32).numpy(),
                                             gain=None if gain is None else gain.numpy())
    xq, s = bl.bitlinear_rmsnorm_quant_act(X.cuda(), gain=None if gain is None else gain.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(xq.cpu().numpy(), xq_ref), "codes must be bit-exact"
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32)), "s must be bit-exact"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("K", [2, 16, 4096])
def test_rmsnorm_quant_act_near_tie(bl, dtype, K):
    """x = [2, 1, 2, 1, ...] with eps = 2^-9: normalising first gives the
    codes 127, 63 (x_n[1] * s = 63.4999962); quantising x and moving the RMS
    factor into s would give 127, 64.  K = 2 takes the element-wise path."""
    X = torch.tensor([2.0, 1.0] * (K // 2)).reshape(1, K).to(dtype)
    xq_ref, s_ref = oracle.rmsnorm_quant_act(X.to(torch.float32).numpy(), eps=np.float32(2.0**-9))
    assert xq_ref[0, :2].tolist() == [127, 63]
    xq, s = bl.bitlinear_rmsnorm_quant_act(X.cuda(), eps=2.0**-9)
    torch.cuda.synchronize()
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))


def test_rmsnorm_quant_act_mixed_exponents_exact_mean(bl):
    """rows whose squares span the whole fp32 range (where any float sum of
    squares drops bits): the exact mean decides r, and a tie of the mean
    (297^2 + 5785^2 = 2 (2^24 + 1)) rounds to even"""
    rows = [[297.0, 5785.0] * 8,
            [1.8e19, 1.0, 1e-20, -2.5e-38, 1e-45, 7.0, -1e10, 5e-3] * 2,
            [3.0e-39, -1e-44, 2.0**-75, 0.0] * 4]
    X = torch.tensor(rows, dtype=torch.float32)
    for eps in (1e-5, 2.0**-100):
        xq_ref, s_ref = oracle.rmsnorm_quant_act(X.numpy(), eps=np.float32(eps))
        xq, s = bl.bitlinear_rmsnorm_quant_act(X.cuda(), eps=eps)
        torch.cuda.synchronize()
        assert np.array_equal(xq.cpu().numpy(), xq_ref)
        assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("M", [3, 600])
def test_rmsnorm_quant_act_unaligned(bl, dtype, M):
    """gain and X views that are not 16-byte aligned take the element-wise path
    (with many tokens too)"""
    K = 1024
    g = torch.Generator().manual_seed(5 + M)
    Xb = (torch.randn((M * K + 1,), generator=g) * 2.0).to(dtype)
    gb = torch.rand((K + 1,), generator=g) + 0.5
    X = Xb[1:].view(M, K)  # starts one element in
    gain = gb[1:]
    xq_ref, s_ref = oracle.rmsnorm_quant_act(X.to(torch.float32).numpy(), gain=gain.numpy())
    xq, s = bl.bitlinear_rmsnorm_quant_act(Xb.cuda()[1:].view(M, K), gain=gb.cuda()[1:])
    torch.cuda.synchronize()
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("M", [256, 1000, 1537, 2051])
@pytest.mark.parametrize("K", [16, 2560, 6912])
@pytest.mark.parametrize("with_gain", [False, True])
def test_rmsnorm_quant_act_many_tokens(bl, dtype, M, K, with_gain):
    """many tokens, special rows (zero, squares overflowing and underflowing
    fp32, large) spread over different CTAs; from 1536 tokens with rows of at
    most 8 KB one warp per row (M = 1537 and 2051 leave the last CTA one and
    three rows)"""
    g = torch.Generator().manual_seed(M + K + with_gain)
    X = torch.randn((M, K), generator=g) * 3.0
    for r, f in ((0, 0.0), (M // 3, 1e30), (M // 2, 1e-40), (M - 1, 1e4)):
        X[r] = X[r] * f
    X = X.to(dtype)
    gain = (torch.rand((K,), generator=g) * 2.0).to(torch.float32) if with_gain else None
    xq_ref, s_ref = oracle.rmsnorm_quant_act(X.to(torch.float32).numpy(),
                                             gain=None if gain is None else gain.numpy())
    xq, s = bl.bitlinear_rmsnorm_quant_act(X.cuda(), gain=None if gain is None else gain.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(xq.cpu().numpy(), xq_ref), "codes must be bit-exact"
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    bl.bitlinear_check_device_error()


def _relu2_case(bl, M, N, K, ws):
    rng = np.random.default_rng(M * 31 + N)
    q = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    p = oracle.pack(q)
    X = torch.randn((M, K), generator=torch.Generator().manual_seed(M + N)).to(torch.bfloat16)
    xq_ref, s_ref = oracle.quant_act(X.to(torch.float32).numpy())
    y_ref, acc_ref = oracle.forward(p, np.float32(0.05), xq_ref, s_ref, K)
    y_ref = oracle.relu2(y_ref)
    call = bl.bitlinear_quant_forward_ws if ws else bl.bitlinear_quant_forward
    y, xq, s, acc = call(torch.from_numpy(p).cuda(), torch.tensor([0.05]).cuda(), X.cuda(), acc=True,
                         flags=bl.BITLINEAR_RELU2)
    torch.cuda.synchronize()
    assert np.array_equal(acc.cpu().numpy(), acc_ref), "acc keeps the raw integer products"
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y_ref.view(np.uint32))
    bl.bitlinear_check_device_error()


@pytest.mark.parametrize("M,N,K", [(1, 300, 1024), (4, 999, 2560), (5, 257, 640), (64, 1000, 2560),
                                   (300, 19000, 128)])
@pytest.mark.parametrize("ws", [False, True])
def test_relu2_epilogue_every_path(bl, M, N, K, ws):
    _relu2_case(bl, M, N, K, ws)


@pytest.mark.parametrize("M", [1, 16])
def test_ffn_chain(bl, M):
    """up projection with the squared ReLU, sub-layer RMS norm + quantisation,
    down projection: the BitNet b1.58 FFN, each step on the GPU."""
    rng = np.random.default_rng(M)
    D, H = 512, 1536
    q_up = rng.integers(-1, 2, size=(H, D)).astype(np.int8)
    q_dn = rng.integers(-1, 2, size=(D, H)).astype(np.int8)
    p_up, p_dn = oracle.pack(q_up), oracle.pack(q_dn)
    g_up, g_dn = np.float32(0.03), np.float32(0.02)
    gain = (rng.uniform(0.5, 1.5, size=H)).astype(np.float32)
    X = torch.randn((M, D), generator=torch.Generator().manual_seed(7)).to(torch.bfloat16)
    # oracle chain
    xq, s = oracle.quant_act(X.to(torch.float32).numpy())
    h, _ = oracle.forward(p_up, g_up, xq, s, D)
    h = oracle.relu2(h)
    hq, hs = oracle.rmsnorm_quant_act(h, gain=gain)
    y_ref, _ = oracle.forward(p_dn, g_dn, hq, hs, H)
    # GPU chain
    dev = "cuda"
    hd, _, _ = bl.bitlinear_quant_forward_ws(torch.from_numpy(p_up).to(dev), torch.tensor([g_up]).to(dev),
                                             X.to(dev), flags=bl.BITLINEAR_RELU2)
    hqd, hsd = bl.bitlinear_rmsnorm_quant_act(hd, gain=torch.from_numpy(gain).to(dev))
    y = bl.bitlinear_forward_ws(torch.from_numpy(p_dn).to(dev), torch.tensor([g_dn]).to(dev), hqd, hsd)
    torch.cuda.synchronize()
    assert np.array_equal(hd.cpu().numpy().view(np.uint32), h.view(np.uint32))
    assert np.array_equal(hqd.cpu().numpy(), hq)
    yr = y.cpu().numpy()
    nz = y_ref != 0
    assert np.all(yr[~nz] == 0)
    assert (np.abs(yr[nz] - y_ref[nz]) / np.abs(y_ref[nz])).max() <= Y_RTOL
    bl.bitlinear_check_device_error()


@pytest.mark.parametrize("M,N,K", [(1, 300, 1024), (4, 999, 2560), (16, 1000, 2560), (64, 700, 8192 + 64),
                                   (97, 2000, 640), (176, 3000, 8192), (300, 19000, 128), (1030, 500, 6912),
                                   (2051, 300, 640)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("with_gain,relu2", [(False, False), (True, True)])
def test_rmsnorm_quant_forward_ws_every_path(bl, M, N, K, dtype, with_gain, relu2):
    """the FFN's second BitLinear in one call, on each route (GEMV after the
    normalising kernel; the normalising kernel writing the fp8 GEMM's split
    operand, or the fp16 operand of the stream-K or persistent GEMM, from 1536
    tokens with short rows one warp per row): x_q and s
    bit-exact against the oracle's RMS-norm quantisation, acc and y bit-exact
    against the oracle's forward on them; special rows included"""
    rng = np.random.default_rng(M * 7 + N + K)
    q = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    p = oracle.pack(q)
    g = torch.Generator().manual_seed(M + K)
    X = torch.randn((M, K), generator=g) * 3.0
    X[0] = 0.0  # an all-zero token
    if M > 2:
        X[M // 2] *= 1e30  # squares overflow fp32: r = inf, codes 0
        X[M - 1] *= 1e-40
    X = X.to(dtype)
    gain = (torch.rand((K,), generator=g) * 2.0).to(torch.float32) if with_gain else None
    xq_ref, s_ref = oracle.rmsnorm_quant_act(X.to(torch.float32).numpy(), gain=None if gain is None else gain.numpy())
    y_ref, acc_ref = oracle.forward(p, np.float32(0.04), xq_ref, s_ref, K, omp=True)
    if relu2:
        y_ref = oracle.relu2(y_ref)
    y, xq, s, acc = bl.bitlinear_rmsnorm_quant_forward_ws(
        torch.from_numpy(p).cuda(), torch.tensor([0.04]).cuda(), X.cuda(),
        gain=None if gain is None else gain.cuda(), acc=True, flags=bl.BITLINEAR_RELU2 if relu2 else 0)
    torch.cuda.synchronize()
    assert np.array_equal(xq.cpu().numpy(), xq_ref), "codes must be bit-exact"
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32)), "s must be bit-exact"
    assert np.array_equal(acc.cpu().numpy(), acc_ref)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y_ref.view(np.uint32))
    bl.bitlinear_check_device_error()


@pytest.mark.parametrize("M", [1, 16, 176])
def test_ffn_chain_one_call_second_bitlinear(bl, M):
    """the down projection through bitlinear_rmsnorm_quant_forward_ws equals
    the two-call chain (bitlinear_rmsnorm_quant_act, then bitlinear_forward_ws)
    bit for bit"""
    rng = np.random.default_rng(100 + M)
    D, H = 512, 1536
    p_up = oracle.pack(rng.integers(-1, 2, size=(H, D)).astype(np.int8))
    p_dn = oracle.pack(rng.integers(-1, 2, size=(D, H)).astype(np.int8))
    gain = torch.from_numpy(rng.uniform(0.5, 1.5, size=H).astype(np.float32)).cuda()
    X = torch.randn((M, D), generator=torch.Generator().manual_seed(9)).to(torch.bfloat16).cuda()
    Wu, Wd = torch.from_numpy(p_up).cuda(), torch.from_numpy(p_dn).cuda()
    gu, gd = torch.tensor([0.03]).cuda(), torch.tensor([0.02]).cuda()
    h, _, _ = bl.bitlinear_quant_forward_ws(Wu, gu, X, flags=bl.BITLINEAR_RELU2)
    hq, hs = bl.bitlinear_rmsnorm_quant_act(h, gain=gain)
    y2 = bl.bitlinear_forward_ws(Wd, gd, hq, hs)
    y1, hq1, hs1 = bl.bitlinear_rmsnorm_quant_forward_ws(Wd, gd, h, gain=gain)
    torch.cuda.synchronize()
    assert torch.equal(hq1, hq)
    assert torch.equal(hs1.view(torch.int32), hs.view(torch.int32))
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))
    bl.bitlinear_check_device_error()


@pytest.mark.parametrize("M,N,K", [(1, 300, 1024), (4, 999, 2560), (3, 260, 40000), (16, 1000, 2560),
                                   (64, 700, 8192 + 64), (97, 2002, 640), (176, 3000, 8192), (2048, 4800, 128)])
@pytest.mark.parametrize("relu2", [False, True])
def test_quant_forward_requant_every_path(bl, M, N, K, relu2):
    """y quantised for the next BitLinear in the same call, on each route (fused GEMV; fp8 GEMM, also for a few tokens
    with K past the GEMV's limit; stream-K GEMM; persistent GEMM): y_q and s_y
    bit-exact against the oracle's per-token quantisation of the oracle's y;
    y, x_q and s bit-exact too.  Rows: an all-zero token (clamped scale), a
    large one and a tiny one whose squared output underflows to zero."""
    rng = np.random.default_rng(M * 11 + N + K)
    p = oracle.pack(rng.integers(-1, 2, size=(N, K)).astype(np.int8))
    X = torch.randn((M, K), generator=torch.Generator().manual_seed(M + 3 * K)) * 2.0
    X[0] = 0.0
    if M > 2:
        X[M // 2] *= 1e12
        X[M - 1] *= 1e-30
    X = X.to(torch.bfloat16)
    xq_ref, s_ref = oracle.quant_act(X.to(torch.float32).numpy(), omp=True)
    y_ref, _ = oracle.forward(p, np.float32(0.05), xq_ref, s_ref, K, omp=True)
    if relu2:
        y_ref = oracle.relu2(y_ref)
    yq_ref, sy_ref = oracle.quant_act(y_ref, omp=True)
    y, xq, s, yq, sy = bl.bitlinear_quant_forward_requant_ws(torch.from_numpy(p).cuda(), torch.tensor([0.05]).cuda(),
                                                             X.cuda(), flags=bl.BITLINEAR_RELU2 if relu2 else 0)
    torch.cuda.synchronize()
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y_ref.view(np.uint32))
    assert np.array_equal(sy.cpu().numpy().view(np.uint32), sy_ref.view(np.uint32)), "s_y must be bit-exact"
    assert np.array_equal(yq.cpu().numpy(), yq_ref), "y_q must be bit-exact"
    bl.bitlinear_check_device_error()


@pytest.mark.parametrize("M", [1, 16, 176])
def test_ffn_chain_requant_feeds_second_bitlinear(bl, M):
    """the up projection's squared-ReLU output quantised in its own call feeds
    the down projection's bitlinear_forward_ws and gives the y of the chain
    that quantises h in a separate bitlinear_quant_act call, bit for bit"""
    rng = np.random.default_rng(300 + M)
    D, H = 512, 1536
    Wu = torch.from_numpy(oracle.pack(rng.integers(-1, 2, size=(H, D)).astype(np.int8))).cuda()
    Wd = torch.from_numpy(oracle.pack(rng.integers(-1, 2, size=(D, H)).astype(np.int8))).cuda()
    gu, gd = torch.tensor([0.03]).cuda(), torch.tensor([0.02]).cuda()
    X = torch.randn((M, D), generator=torch.Generator().manual_seed(11)).to(torch.bfloat16).cuda()
    h, _, _ = bl.bitlinear_quant_forward_ws(Wu, gu, X, flags=bl.BITLINEAR_RELU2)
    hq, hs = bl.bitlinear_quant_act(h)
    y2 = bl.bitlinear_forward_ws(Wd, gd, hq, hs)
    h1, _, _, hq1, hs1 = bl.bitlinear_quant_forward_requant_ws(Wu, gu, X, flags=bl.BITLINEAR_RELU2)
    y1 = bl.bitlinear_forward_ws(Wd, gd, hq1, hs1)
    torch.cuda.synchronize()
    assert torch.equal(h1.view(torch.int32), h.view(torch.int32))
    assert torch.equal(hq1, hq)
    assert torch.equal(hs1.view(torch.int32), hs.view(torch.int32))
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))
    bl.bitlinear_check_device_error()
