"""The tcgen05 symmetric GEMM through the C ABI against a plain fp64 product of
the same fp16 inputs (Dion3 §5: D = alpha A B + beta C with symmetric results,
lower-triangle tiles mirrored into the upper triangle)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gns():
    import newton_schulz_gram_gb300 as m
    from newton_schulz_gram_gb300 import build
    build.build()
    m.load()
    return m


def _half(a):
    return np.asarray(a, np.float32).astype(np.float16)


@pytest.mark.parametrize("G,n,k", [(1, 128, 64), (1, 128, 512), (2, 256, 192), (3, 200, 136), (1, 384, 1000),
                                   (2, 8, 16), (1, 520, 72)])
def test_gram_product(gns, G, n, k):
    rng = np.random.default_rng(n * 7 + k)
    A = _half(rng.standard_normal((G, n, k)) / np.sqrt(k))
    dev = torch.device("cuda")
    tA = torch.from_numpy(A).to(dev)
    tD = torch.full((G, n, n), float("nan"), dtype=torch.float16, device=dev)
    gns.gns_symm_gemm(tA, tA, None, tD, alpha=1.0, beta=0.0)
    torch.cuda.synchronize()
    D = tD.cpu().numpy()
    ref = np.einsum("gik,gjk->gij", A.astype(np.float64), A.astype(np.float64))
    assert np.all(np.isfinite(D)), "some output element was never written"
    for g in range(G):
        assert np.array_equal(D[g], D[g].T), "output not exactly symmetric"
        err = np.abs(D[g].astype(np.float64) - ref[g]).max()
        assert err <= 2e-3 * np.abs(ref[g]).max() + 1e-3, err


@pytest.mark.parametrize("G,n", [(1, 128), (2, 256), (1, 200), (3, 136)])
def test_symmetric_product_with_addend(gns, G, n):
    rng = np.random.default_rng(n)
    S = rng.standard_normal((G, n, n))
    S = (S + S.transpose(0, 2, 1)) / (2 * np.sqrt(n))
    T = rng.standard_normal((G, n, n))
    T = (T + T.transpose(0, 2, 1)) / (2 * np.sqrt(n))
    Ah, Bh = _half(S), _half(T)
    C = _half(rng.standard_normal((G, n, n)))
    C = _half((C.astype(np.float32) + C.astype(np.float32).transpose(0, 2, 1)) / 2)
    dev = torch.device("cuda")
    tD = torch.full((G, n, n), float("nan"), dtype=torch.float16, device=dev)
    alpha, beta = 0.75, -1.5
    gns.gns_symm_gemm(torch.from_numpy(Ah).to(dev), torch.from_numpy(Bh).to(dev), torch.from_numpy(C).to(dev),
                      tD, alpha=alpha, beta=beta)
    torch.cuda.synchronize()
    D = tD.cpu().numpy().astype(np.float64)
    # Lower triangle is alpha A B^T + beta C (B symmetric, so B^T = B).
    ref = alpha * np.einsum("gik,gjk->gij", Ah.astype(np.float64), Bh.astype(np.float64)) + beta * C.astype(np.float64)
    for g in range(G):
        low = np.tril_indices(n)
        err = np.abs(D[g][low] - ref[g][low]).max()
        assert err <= 2e-3 * np.abs(ref[g]).max() + 2e-3, err
        assert np.array_equal(D[g], D[g].T)
