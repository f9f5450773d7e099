"""tcgen05 GEMM (dion3_gemm_f16) against numpy float64 products of the same
fp16 operands.  Shapes span several 128 x 128 tiles with ragged tails."""
import numpy as np
import pytest
import torch

import matrix_orthogonalizing_optimizer_shape_gb300 as d3
from tests._harness import rel_fro

pytestmark = pytest.mark.gpu


def _h(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to("cuda").half()


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


def _padded(rows, cols, batch=1, pad_to=8, fill=0.0):
    ld = (cols + pad_to - 1) // pad_to * pad_to
    return torch.full((batch, rows, ld), fill, dtype=torch.float16, device="cuda")


@pytest.mark.parametrize("s,L", [(64, 64), (128, 64), (200, 136), (256, 1024), (333, 700), (520, 96)])
def test_syrk_lower_mirrored(cuda_lib, s, L):
    rng = np.random.default_rng(s * 1000 + L)
    A = rng.standard_normal((s, L)) / np.sqrt(L)
    Ad = _padded(s, L)
    Ad[0, :, :L] = _h(A)
    D = _padded(s, s, fill=float("nan"))
    d3.gemm_f16(Ad[:, :, :L], Ad[:, :, :L], D=D[:, :, :s], mode=d3.GEMM_SYM_LOWER)
    torch.cuda.synchronize()
    got = _np(D[0, :, :s])
    A16 = _np(Ad[0, :, :L])
    want = A16 @ A16.T
    assert np.isfinite(got).all()
    assert np.array_equal(got, got.T)  # exactly symmetric by construction
    assert rel_fro(got, want) < 2e-3


@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (300, 136, 200), (1000, 256, 256), (77, 300, 520)])
def test_rect_normal_and_transposed(cuda_lib, M, N, K):
    rng = np.random.default_rng(M + N + K)
    A = rng.standard_normal((M, K)) / np.sqrt(K)
    B = rng.standard_normal((N, K))
    Ad, Bd = _padded(M, K), _padded(N, K)
    Ad[0, :, :K] = _h(A)
    Bd[0, :, :K] = _h(B)
    D = _padded(M, N, fill=float("nan"))
    DT = _padded(N, M, fill=float("nan"))
    d3.gemm_f16(Ad[:, :, :K], Bd[:, :, :K], D=D[:, :, :N], DT=DT[:, :, :M], mode=d3.GEMM_RECT)
    torch.cuda.synchronize()
    want = _np(Ad[0, :, :K]) @ _np(Bd[0, :, :K]).T
    got, gotT = _np(D[0, :, :N]), _np(DT[0, :, :M])
    assert np.isfinite(got).all() and np.array_equal(gotT, got.T)
    assert rel_fro(got, want) < 2e-3


@pytest.mark.parametrize("s", [96, 256, 300])
def test_polynomial_epilogue_batched(cuda_lib, s):
    # Z = c R.R + b R + a I for a batch of symmetric R (the NS polynomial step).
    a, b, c = d3.MUON_QUINTIC
    rng = np.random.default_rng(s)
    batch = 3
    Rs = []
    for _ in range(batch):
        X = rng.standard_normal((s, 2 * s))
        X /= np.linalg.norm(X)
        Rs.append(X @ X.T)
    Rd = _padded(s, s, batch)
    for i, R in enumerate(Rs):
        Rd[i, :, :s] = _h(R)
    Zd = _padded(s, s, batch, fill=float("nan"))
    d3.gemm_f16(Rd[:, :, :s], Rd[:, :, :s], D=Zd[:, :, :s], C=Rd[:, :, :s], mode=d3.GEMM_SYM_LOWER,
                alpha=c, beta=b, gamma=a)
    torch.cuda.synchronize()
    for i in range(batch):
        R16 = _np(Rd[i, :, :s])
        want = c * R16 @ R16 + b * R16 + a * np.eye(s)
        got = _np(Zd[i, :, :s])
        assert np.array_equal(got, got.T)
        assert rel_fro(got, want) < 2e-3


def test_batch_stride_isolation(cuda_lib):
    # Each matrix of a batch uses only its own operands.
    s, L, batch = 130, 200, 4
    rng = np.random.default_rng(1)
    Ad = _padded(s, L, batch)
    for i in range(batch):
        Ad[i, :, :L] = _h(rng.standard_normal((s, L)) * (i + 1) / np.sqrt(L))
    D = _padded(s, s, batch, fill=float("nan"))
    d3.gemm_f16(Ad[:, :, :L], Ad[:, :, :L], D=D[:, :, :s], mode=d3.GEMM_SYM_LOWER)
    torch.cuda.synchronize()
    for i in range(batch):
        A16 = _np(Ad[i, :, :L])
        assert rel_fro(_np(D[i, :, :s]), A16 @ A16.T) < 2e-3
    d3.device_status()
