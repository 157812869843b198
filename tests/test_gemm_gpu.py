"""The library's internal GEMMs (tcgen05 and SIMT) checked element by element
against an fp64 CPU product of the same (bf16-exact) inputs, through the
rnn_debug_gemm hook: K-major and MN-major operands, ragged M / N / K tails,
bias, accumulate-into-C, bf16 output and the gate-slot row remap."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


def _lib():
    from bwd_persistent_cta_gb300 import build
    build.build()
    import bwd_persistent_cta_gb300 as R
    return R


def _case(M, N, K, a_kmajor, b_kmajor, use_tc, bias=False, beta=False, c_bf16=False, rowmap=None, seed=0):
    R = _lib()
    g = torch.Generator().manual_seed(seed)
    dt = torch.bfloat16 if use_tc else torch.float32
    Am = torch.randn(M, K, generator=g).to(dt)
    Bm = torch.randn(N, K, generator=g).to(dt)
    A_store = Am if a_kmajor else Am.t().contiguous()
    B_store = Bm if b_kmajor else Bm.t().contiguous()
    lda = K if a_kmajor else M
    ldb = K if b_kmajor else N
    ref = Am.double() @ Bm.double().t()
    bias_t = torch.randn(N, generator=g) if bias else None
    if bias:
        ref = ref + bias_t.double()[None, :]
    H = M // 4 if rowmap else 0
    perm = rowmap or [0, 1, 2, 3]
    out_rows = M
    C0 = torch.randn(out_rows, N, generator=g)
    if c_bf16:
        C0 = C0.bfloat16().float()
    # expected output rows
    exp = C0.double().clone()
    for m in range(M):
        row = m
        if rowmap:
            p = perm[m & 3]
            if p < 0:
                continue
            row = p * H + (m >> 2)
        exp[row] = ref[m] + (C0.double()[row] if beta else 0.0)
    Cd = C0.to("cuda", torch.bfloat16 if c_bf16 else torch.float32)
    Ad, Bd = A_store.cuda(), B_store.cuda()          # kept alive until the kernel has run
    biasd = bias_t.cuda() if bias else None
    rc = R.rnn_debug_gemm(M, N, K, Ad.data_ptr(), lda, int(a_kmajor), Bd.data_ptr(), ldb,
                          int(b_kmajor), Cd.data_ptr(), N, int(c_bf16),
                          biasd.data_ptr() if bias else None, int(beta), H, perm, int(use_tc), int(use_tc),
                          torch.cuda.current_stream().cuda_stream)
    assert rc == 0, R.rnn_status_string(rc)
    torch.cuda.synchronize()
    got = Cd.double().cpu()
    scale = float(exp.abs().max())
    err = float((got - exp).abs().max()) / scale
    # fp32 output: the tensor cores' fp32 accumulation error grows with the
    # length of one accumulation chain (an unsplit K = 8192 reaches ~1.1e-5 of
    # the largest output), so the bound is 1e-5 up to K = 4096, then linear in K
    tol = 1e-2 if c_bf16 else (2e-5 if not use_tc else 1e-5 * max(1.0, K / 4096))
    assert err < tol, (err, M, N, K, a_kmajor, b_kmajor, use_tc)


@pytest.mark.parametrize("use_tc", [1, 0])
@pytest.mark.parametrize("a_kmajor,b_kmajor", [(1, 1), (0, 0), (1, 0), (0, 1)])
def test_gemm_layouts(use_tc, a_kmajor, b_kmajor):
    _case(256, 384, 192, a_kmajor, b_kmajor, use_tc)


@pytest.mark.parametrize("use_tc", [1, 0])
@pytest.mark.parametrize("M,N,K", [(200, 136, 72), (128, 128, 64), (1000, 264, 520), (8, 16, 8)])
def test_gemm_ragged(use_tc, M, N, K):
    _case(M, N, K, 1, 1, use_tc, seed=M + N + K)


@pytest.mark.parametrize("use_tc", [1, 0])
def test_gemm_epilogue_bias_bf16(use_tc):
    _case(384, 256, 128, 1, 1, use_tc, bias=True, c_bf16=True)


@pytest.mark.parametrize("use_tc", [1, 0])
def test_gemm_epilogue_beta_rowmap(use_tc):
    _case(512, 200, 1000, 0, 0, use_tc, beta=True, rowmap=[2, 0, -1, 1])


@pytest.mark.parametrize("use_tc", [1, 0])
def test_gemm_epilogue_bf16_beta_bias_rowmap_ragged(use_tc):
    # bf16 output with accumulate, bias and the row remap; N = 8 full 32-column chunks + 8
    _case(384, 264, 200, 1, 1, use_tc, bias=True, beta=True, c_bf16=True, rowmap=[3, -1, 0, 1], seed=14)


@pytest.mark.parametrize("use_tc", [1, 0])
def test_gemm_epilogue_f32_bias(use_tc):
    _case(200, 96, 64, 1, 0, use_tc, bias=True, seed=15)


def test_gemm_split_k_rowmap_beta_bias():
    # long K, few tiles: K is split across CTAs; the partials are summed in split order
    _case(512, 512, 8192, 0, 0, 1, bias=True, beta=True, rowmap=[1, -1, 0, 2], seed=11)


@pytest.mark.parametrize("splits", [2, 3])
def test_gemm_split_k_multiwave(plan_overrides, splits):
    # more (tile, split) items than SMs (a forced split): the split items run
    # in several waves, each split of a tile after the one before it
    plan_overrides(gemm_splits=splits)
    _case(6400, 512, 3072, 1, 1, 1, seed=12)


def test_gemm_split_k_deterministic():
    R = _lib()
    g = torch.Generator().manual_seed(13)
    M, N, K = 1024, 512, 16384
    A = torch.randn(M, K, generator=g).bfloat16().cuda()
    B = torch.randn(N, K, generator=g).bfloat16().cuda()
    outs = []
    for _ in range(2):
        C = torch.zeros(M, N, device="cuda")
        rc = R.rnn_debug_gemm(M, N, K, A.data_ptr(), K, 1, B.data_ptr(), K, 1, C.data_ptr(), N, 0, None, 0, 0,
                              [0, 1, 2, 3], 1, 1, torch.cuda.current_stream().cuda_stream)
        assert rc == 0, R.rnn_status_string(rc)
        torch.cuda.synchronize()
        outs.append(C.cpu())
    assert torch.equal(outs[0], outs[1])
    ref = A.double().cpu() @ B.double().cpu().t()
    assert float((outs[0].double() - ref).abs().max()) / float(ref.abs().max()) < 1e-5


# 256 x 256 tiles (two M=128 halves sharing each B stage, one accumulator)
@pytest.mark.parametrize("a_kmajor,b_kmajor", [(1, 1), (0, 0), (1, 0), (0, 1)])
def test_gemm_tall_tiles_layouts(plan_overrides, a_kmajor, b_kmajor):
    plan_overrides(gemm_tm=256)
    _case(512, 512, 320, a_kmajor, b_kmajor, 1, seed=20 + 2 * a_kmajor + b_kmajor)


@pytest.mark.parametrize("M,N,K", [(200, 136, 72), (1000, 264, 520), (300, 700, 64), (8, 16, 8)])
def test_gemm_tall_tiles_ragged(plan_overrides, M, N, K):
    plan_overrides(gemm_tm=256)
    _case(M, N, K, 1, 1, 1, seed=30 + M + N + K)


def test_gemm_tall_tiles_epilogue(plan_overrides):
    plan_overrides(gemm_tm=256)
    _case(640, 264, 200, 1, 1, 1, bias=True, beta=True, c_bf16=True, rowmap=[3, -1, 0, 1], seed=41)
    _case(512, 200, 1000, 0, 0, 1, beta=True, rowmap=[2, 0, -1, 1], seed=42)


@pytest.mark.parametrize("splits", [1, 2, 3])
def test_gemm_tall_tiles_split_k(plan_overrides, splits):
    # more (tile, split) items than SMs at split 2 and 3
    plan_overrides(gemm_tm=256, gemm_splits=splits)
    _case(12800, 768, 3072, 1, 1, 1, seed=43 + splits)
    _case(512, 512, 8192, 0, 0, 1, bias=True, beta=True, rowmap=[1, -1, 0, 2], seed=47)


@pytest.mark.parametrize("tm", [128, 256])
@pytest.mark.parametrize("M,N,K", [(300, 200, 128), (260, 196, 96), (384, 520, 4096)])
def test_gemm_bf16_output_ragged_rows(plan_overrides, tm, M, N, K):
    # bf16 output without accumulate (whole 128-byte row segments, a scalar
    # tail where N ends inside a segment or rows are not 16-byte aligned)
    plan_overrides(gemm_tm=tm)
    _case(M, N, K, 1, 1, 1, bias=True, c_bf16=True, seed=M + N)
    # MN-major A where its rows stay 16-byte aligned (M a multiple of 8)
    _case(M, N, K, int(M % 8 != 0), 1, 1, c_bf16=True, rowmap=[1, 3, -1, 0], seed=M + N + 1)
