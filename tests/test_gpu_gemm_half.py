"""Half-stored symmetric matrices in the tcgen05 GEMM (the DION3_GEMM_*_HALF
mode flags): only the 256 x 256 blocks below the block diagonal and the full
diagonal blocks hold values.  Products that read such operands (the K ranges
above the diagonal come from the transpose, as MN-major tiles) must equal the
products of the fully stored matrices; the region above the diagonal blocks is
filled with NaN so that any read of it shows.  A half-stored result must equal
the full result wherever it is defined, and leave the rest untouched."""
import numpy as np
import pytest
import torch

import matrix_orthogonalizing_optimizer_shape_gb300 as d3
from tests._harness import rel_fro

pytestmark = pytest.mark.gpu

SYM_HALF = d3.GEMM_SYM_LOWER | d3.GEMM_OUT_HALF | d3.GEMM_A_HALF | d3.GEMM_B_HALF


def _half_mask(s):
    """True where a half-stored s x s matrix is defined."""
    blk = np.arange(s) // 256
    return blk[:, None] >= blk[None, :]


def _sym(rng, batch, s, scale):
    x = rng.standard_normal((batch, s, s)) * scale
    return (x + np.swapaxes(x, 1, 2)) / 2


def _dev(x, ld=None):
    b, r, c = x.shape
    ld = ld or (c + 7) // 8 * 8
    t = torch.full((b, r, ld), float("nan"), dtype=torch.float16, device="cuda")
    t[:, :, :c] = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to("cuda").half()
    return t


def _as_half_stored(t, s):
    """The same device matrices with NaN outside the half-stored region."""
    h = t.clone()
    m = torch.from_numpy(~_half_mask(s)).to("cuda")
    h[:, :s, :s][:, m] = float("nan")
    return h


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("s,batch", [(200, 3), (256, 2), (512, 2), (700, 2), (1024, 1)])
def test_half_operands_and_output_match_full(cuda_lib, s, batch):
    rng = np.random.default_rng(s + 17 * batch)
    R = _dev(_sym(rng, batch, s, 1.0 / np.sqrt(s)))
    Cm = _dev(_sym(rng, batch, s, 0.3))
    a, b, c = d3.MUON_QUINTIC
    full = _dev(np.zeros((batch, s, s)))
    d3.gemm_f16(R[:, :, :s], R[:, :, :s], D=full[:, :, :s], C=Cm[:, :, :s], mode=d3.GEMM_SYM_LOWER,
                alpha=c, beta=b, gamma=a)
    Rh, Ch = _as_half_stored(R, s), _as_half_stored(Cm, s)
    out = _dev(np.full((batch, s, s), 7.0))
    d3.gemm_f16(Rh[:, :, :s], Rh[:, :, :s], D=out[:, :, :s], C=Ch[:, :, :s], mode=SYM_HALF,
                alpha=c, beta=b, gamma=a)
    torch.cuda.synchronize()
    mask = _half_mask(s)
    got, ref = _np(out[:, :, :s]), _np(full[:, :, :s])
    assert np.isfinite(got[:, mask]).all()
    # Same fp16 operand values, same accumulation: the results agree to the
    # last bit or within a few fp16 ulps.
    assert np.abs(got[:, mask] - ref[:, mask]).max() <= 4e-3 * max(1.0, np.abs(ref).max())
    # Outside the diagonal blocks nothing above them was written.
    assert (got[:, ~mask] == 7.0).all()
    # The diagonal blocks are exactly symmetric.
    for b0 in range(0, s, 256):
        blk = got[:, b0:b0 + 256, b0:b0 + 256]
        assert np.array_equal(blk, np.swapaxes(blk, 1, 2))
    # And against float64 on the fp16 operands.
    R64, C64 = _np(R[:, :, :s]), _np(Cm[:, :, :s])
    want = c * R64 @ R64 + b * C64 + a * np.eye(s)
    assert rel_fro(np.where(mask, got, 0), np.where(mask, want, 0)) < 2e-3


@pytest.mark.parametrize("L,s,batch", [(1000, 520, 2), (4096, 1024, 1), (300, 700, 2)])
def test_rect_with_half_stored_b(cuda_lib, L, s, batch):
    rng = np.random.default_rng(L + s)
    Yt = _dev(rng.standard_normal((batch, L, s)) / np.sqrt(s))
    Q = _dev(_sym(rng, batch, s, 1.0 / np.sqrt(s)))
    D1 = _dev(np.zeros((batch, L, s)))
    DT1 = _dev(np.zeros((batch, s, L)))
    d3.gemm_f16(Yt[:, :, :s], Q[:, :, :s], D=D1[:, :, :s], DT=DT1[:, :, :L], mode=d3.GEMM_RECT)
    Qh = _as_half_stored(Q, s)
    D2 = _dev(np.zeros((batch, L, s)))
    DT2 = _dev(np.zeros((batch, s, L)))
    d3.gemm_f16(Yt[:, :, :s], Qh[:, :, :s], D=D2[:, :, :s], DT=DT2[:, :, :L],
                mode=d3.GEMM_RECT | d3.GEMM_B_HALF)
    torch.cuda.synchronize()
    g1, g2 = _np(D1[:, :, :s]), _np(D2[:, :, :s])
    assert np.isfinite(g2).all()
    assert np.abs(g2 - g1).max() <= 4e-3 * max(1.0, np.abs(g1).max())
    assert np.array_equal(_np(DT2[:, :, :L]), np.swapaxes(g2, 1, 2))
    want = _np(Yt[:, :, :s]) @ _np(Q[:, :, :s])
    assert rel_fro(g2, want) < 2e-3


def test_half_flag_rules(cuda_lib):
    A = torch.zeros((1, 256, 128), dtype=torch.float16, device="cuda")
    D = torch.zeros((1, 256, 256), dtype=torch.float16, device="cuda")
    with pytest.raises(d3.Dion3Error):   # A_HALF needs M == K
        d3.gemm_f16(A, A, D=D, mode=d3.GEMM_SYM_LOWER | d3.GEMM_A_HALF)
    with pytest.raises(d3.Dion3Error):   # OUT_HALF needs the symmetric mode
        d3.gemm_f16(A, A, D=D, mode=d3.GEMM_RECT | d3.GEMM_OUT_HALF)
    with pytest.raises(d3.Dion3Error):   # unknown flag
        d3.gemm_f16(A, A, D=D, mode=d3.GEMM_SYM_LOWER | 0x800)


@pytest.mark.parametrize("M,N,K,batch", [(1000, 520, 520, 2), (300, 700, 1024, 1), (4096, 1024, 1024, 1)])
def test_transposed_operands_match_plain(cuda_lib, M, N, K, batch):
    """A (or B) passed as its transpose, read as MN-major tiles, gives the same
    product as the plain K-major operand."""
    rng = np.random.default_rng(M + 3 * N + 7 * K)
    A = _dev(rng.standard_normal((batch, M, K)) / np.sqrt(K))
    B = _dev(rng.standard_normal((batch, N, K)))
    # The same fp16 values stored transposed (pitches padded to 8 elements).
    At = _dev(np.swapaxes(_np(A[:, :, :K]), 1, 2))[:, :, :M]
    Bt = _dev(np.swapaxes(_np(B[:, :, :K]), 1, 2))[:, :, :N]
    ref = _dev(np.zeros((batch, M, N)))
    d3.gemm_f16(A[:, :, :K], B[:, :, :K], D=ref[:, :, :N])
    for mode, a, b in [(d3.GEMM_A_TRANS, At, B[:, :, :K]), (d3.GEMM_B_TRANS, A[:, :, :K], Bt),
                       (d3.GEMM_A_TRANS | d3.GEMM_B_TRANS, At, Bt)]:
        D = _dev(np.zeros((batch, M, N)))
        DT = _dev(np.zeros((batch, N, M)))
        d3.gemm_f16(a, b, D=D[:, :, :N], DT=DT[:, :, :M], mode=d3.GEMM_RECT | mode)
        torch.cuda.synchronize()
        got, want = _np(D[:, :, :N]), _np(ref[:, :, :N])
        assert np.isfinite(got).all()
        assert np.abs(got - want).max() <= 4e-3 * max(1.0, np.abs(want).max()), mode
        assert np.array_equal(_np(DT[:, :, :M]), np.swapaxes(got, 1, 2))


def test_syrk_from_transposed_storage(cuda_lib):
    """R = Y Y^T with Y given as its transpose (the k > m case of the Gram
    path), written half-stored."""
    rng = np.random.default_rng(5)
    batch, s, L = 2, 700, 1500
    Yt = _dev(rng.standard_normal((batch, L, s)) / np.sqrt(L))      # stored Y^T, [L][s]
    R = _dev(np.full((batch, s, s), 7.0))
    d3.gemm_f16(Yt[:, :, :s], Yt[:, :, :s], D=R[:, :, :s],
                mode=d3.GEMM_SYM_LOWER | d3.GEMM_OUT_HALF | d3.GEMM_A_TRANS | d3.GEMM_B_TRANS)
    torch.cuda.synchronize()
    Y = np.swapaxes(_np(Yt[:, :, :s]), 1, 2)
    want = Y @ np.swapaxes(Y, 1, 2)
    mask = _half_mask(s)
    got = _np(R[:, :, :s])
    assert (got[:, ~mask] == 7.0).all()
    assert rel_fro(np.where(mask, got, 0), np.where(mask, want, 0)) < 2e-3


@pytest.mark.parametrize("s,batch", [(256, 2), (700, 2), (1024, 1)])
@pytest.mark.parametrize("with_c", [False, True])
def test_self_product_diagonal_blocks_whole(cuda_lib, s, batch, with_c):
    """R R^T (+ b R + a I) with A, B and C the same half-stored matrix: the
    diagonal blocks are written whole as computed, not mirrored.  Entry (i, j)
    and (j, i) are the same sum of the same products, so the result equals,
    bit for bit, the mirrored result of the same product with B (and C) in
    another buffer holding the same values."""
    rng = np.random.default_rng(s + batch + 100 * with_c)
    R = _as_half_stored(_dev(_sym(rng, batch, s, 1.0 / np.sqrt(s))), s)
    R2 = R.clone()
    a, b, c = d3.MUON_QUINTIC
    whole = _dev(np.full((batch, s, s), 7.0))
    mirrored = _dev(np.full((batch, s, s), 7.0))
    beta = b if with_c else 0.0
    d3.gemm_f16(R[:, :, :s], R[:, :, :s], D=whole[:, :, :s], C=R[:, :, :s] if with_c else None,
                mode=SYM_HALF, alpha=c, beta=beta, gamma=a)
    d3.gemm_f16(R[:, :, :s], R2[:, :, :s], D=mirrored[:, :, :s], C=R2[:, :, :s] if with_c else None,
                mode=SYM_HALF, alpha=c, beta=beta, gamma=a)
    torch.cuda.synchronize()
    mask = _half_mask(s)
    got, ref = _np(whole[:, :, :s]), _np(mirrored[:, :, :s])
    assert np.isfinite(got[:, mask]).all()
    assert np.array_equal(got[:, mask], ref[:, mask])
    assert (got[:, ~mask] == 7.0).all()
    R64 = np.where(mask, _np(R[:, :, :s]), np.swapaxes(np.nan_to_num(_np(R[:, :, :s])), 1, 2))
    want = c * R64 @ R64 + beta * R64 + a * np.eye(s)
    assert rel_fro(np.where(mask, got, 0), np.where(mask, want, 0)) < 2e-3


@pytest.mark.parametrize("tr", [False, True])
def test_syrk_diagonal_blocks_whole(cuda_lib, tr):
    """Y Y^T written half-stored from one buffer (diagonal blocks whole) equals
    the mirrored result with B in a copy of Y, bit for bit."""
    rng = np.random.default_rng(9 + tr)
    batch, s, L = 2, 600, 1300
    if tr:
        Yf = _dev(rng.standard_normal((batch, L, s)) / np.sqrt(L))
        Y, Y2 = Yf[:, :, :s], Yf.clone()[:, :, :s]
        mode = d3.GEMM_SYM_LOWER | d3.GEMM_OUT_HALF | d3.GEMM_A_TRANS | d3.GEMM_B_TRANS
    else:
        Yf = _dev(rng.standard_normal((batch, s, L)) / np.sqrt(L))
        Y, Y2 = Yf[:, :, :L], Yf.clone()[:, :, :L]
        mode = d3.GEMM_SYM_LOWER | d3.GEMM_OUT_HALF
    whole = _dev(np.full((batch, s, s), 7.0))
    mirrored = _dev(np.full((batch, s, s), 7.0))
    d3.gemm_f16(Y, Y, D=whole[:, :, :s], mode=mode)
    d3.gemm_f16(Y, Y2, D=mirrored[:, :, :s], mode=mode)
    torch.cuda.synchronize()
    mask = _half_mask(s)
    got, ref = _np(whole[:, :, :s]), _np(mirrored[:, :, :s])
    assert np.array_equal(got[:, mask], ref[:, mask])
    assert (got[:, ~mask] == 7.0).all()


@pytest.mark.parametrize("s,L,batch", [(520, 1000, 2), (1024, 4096, 1), (700, 300, 2)])
def test_rect_half_a_with_transposed_b(cuda_lib, s, L, batch):
    """D = Q Y with Q half-stored (A) and B = Y^T passed as its transpose, i.e.
    Y itself (the product that writes O in Y's orientation): equal to the same
    product with Q fully stored and Y^T given explicitly."""
    rng = np.random.default_rng(s + 3 * L)
    Q = _dev(_sym(rng, batch, s, 1.0 / np.sqrt(s)))
    Y = _dev(rng.standard_normal((batch, s, L)))
    Yt = _dev(np.swapaxes(_np(Y[:, :, :L]), 1, 2))
    ref = _dev(np.zeros((batch, s, L)))
    d3.gemm_f16(Q[:, :, :s], Yt[:, :, :s], D=ref[:, :, :L])
    got = _dev(np.zeros((batch, s, L)))
    d3.gemm_f16(_as_half_stored(Q, s)[:, :, :s], Y[:, :, :L], D=got[:, :, :L],
                mode=d3.GEMM_RECT | d3.GEMM_A_HALF | d3.GEMM_B_TRANS)
    torch.cuda.synchronize()
    g, r = _np(got[:, :, :L]), _np(ref[:, :, :L])
    assert np.isfinite(g).all()
    assert np.abs(g - r).max() <= 4e-3 * max(1.0, np.abs(r).max())
    want = _np(Q[:, :, :s]) @ _np(Y[:, :, :L])
    assert rel_fro(g, want) < 2e-3
