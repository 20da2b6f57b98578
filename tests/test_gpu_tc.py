"""The tensor-core GEMM tile (tcgen05 + TMEM + TMA) against the oracle's
linear map on bf16 inputs, with B stored [N][K] (weights) or [K][N] (the V
cache as prefill attention reads it).  Tolerance: f32 accumulation of exact
bf16 products, |C - ref| <= 4e-5 * sqrt(K) * max|A| * max|B| (written here)."""
import numpy as np
import pytest
import torch

import oracle
from tile_level_overlap_gb300 import build, mk, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    mk.lib()


@pytest.mark.parametrize("b_layout", [0, 1])
@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (128, 256, 128), (256, 512, 1024),
                                   (200, 384, 320), (1, 256, 64), (384, 1280, 4096)])
def test_tc_gemm_matches_oracle_linear(M, N, K, b_layout):
    dev = torch.device("cuda:0")
    g = torch.Generator(device="cpu").manual_seed(M * 7 + N * 3 + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g).to(torch.bfloat16)
    Ad = A.to(dev)
    Bd = (B if b_layout == 0 else B.t().contiguous()).to(dev)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    rc = mk.lib().mk_debug_gemm_bf16(Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(), M, N, K, b_layout,
                                     torch.cuda.current_stream().cuda_stream)
    assert rc == mk.MK_OK
    ref = oracle.linear(synth.bf16_bits(B), oracle.widen_bf16(synth.bf16_bits(A)), np.float64)
    got = C.cpu().numpy()
    bound = 4e-5 * np.sqrt(K) * np.abs(A.float().numpy()).max() * np.abs(B.float().numpy()).max()
    err = np.abs(got - ref).max()
    assert err <= bound, f"max |delta| {err:.3e} > {bound:.3e}"


def test_tc_gemm_rejects_bad_shapes():
    L = mk.lib()
    assert L.mk_debug_gemm_bf16(None, None, None, 128, 128, 64, 0, None) == mk.MK_ERR_INVALID_ARG
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    p = x.data_ptr()
    assert L.mk_debug_gemm_bf16(p, p, p, 128, 100, 64, 0, None) == mk.MK_ERR_INVALID_ARG
    assert L.mk_debug_gemm_bf16(p, p, p, 128, 128, 96, 0, None) == mk.MK_ERR_INVALID_ARG
    assert L.mk_debug_gemm_bf16(p, p, p, 128, 128, 64, 2, None) == mk.MK_ERR_INVALID_ARG
