"""Gram Newton-Schulz on the GPU, through the C ABI, against the fp64 oracle
on the same seeded inputs (Dion3 Algorithm 3 for rectangular matrices,
Algorithm 1 for square ones)."""
import numpy as np
import pytest

from gpu_helpers import assert_parity, parity_metrics
from inputs import generators as gen
from oracle import gram_ns as O

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gns():
    import newton_schulz_gram_gb300 as m
    from newton_schulz_gram_gb300 import build
    build.build()
    m.load()
    return m


def run_gpu(gns, X, **kw):
    t = torch.from_numpy(np.ascontiguousarray(X, dtype=np.float32)).cuda()
    gns.gns_orthogonalize_batched(t, **kw)
    torch.cuda.synchronize()
    assert gns.gns_get_status() == 0
    return t.cpu().numpy()


SHAPES = [
    (1, 128, 512),   # the 128 x 512 single-matrix case
    (2, 512, 128),   # transposed orientation
    (3, 200, 712),   # ragged: n, m not multiples of the tiles
    (2, 712, 200),
    (1, 96, 1000),
    (2, 8, 32),
    (1, 1, 7),       # n = 1
    (2, 130, 4100),  # one row past a tile, ragged K
    (2, 256, 256),   # square: standard NS
    (1, 200, 200),   # ragged square
    (4, 384, 1536),
]


@pytest.mark.parametrize("G,R,C", SHAPES)
def test_matches_oracle(gns, G, R, C):
    X = gen.gaussian_bucket(G, R, C, seed=100 + R + C)
    out = run_gpu(gns, X)
    for g in range(G):
        ref = O.orthogonalize(X[g].astype(np.float64))
        assert_parity(out[g], ref, what=f"{R}x{C}[{g}]")


def test_single_128x512_against_both_references(gns):
    """The 128 x 512 case against restarted Gram NS and against standard NS
    (which agree to ~1e-13 in fp64)."""
    X = gen.gaussian_bucket(1, 128, 512, seed=1000)
    out = run_gpu(gns, X)[0]
    assert_parity(out, O.gram_ns(X[0].astype(np.float64)))
    assert_parity(out, O.standard_ns(X[0].astype(np.float64)))


def test_grouped_equals_single_bitwise(gns):
    for R, C in ((256, 1024), (1024, 256), (192, 192)):
        X = gen.gaussian_bucket(5, R, C, seed=7)
        grouped = run_gpu(gns, X)
        for g in range(5):
            single = run_gpu(gns, X[g:g + 1])
            assert np.array_equal(single[0], grouped[g]), (R, C, g)


def test_zero_matrix_gives_zero(gns):
    for shape in ((2, 64, 256), (1, 128, 128)):
        out = run_gpu(gns, np.zeros(shape, np.float32))
        assert np.all(out == 0)


@pytest.mark.parametrize("scale", [1e-3, 1e3])
def test_scaled_inputs(gns, scale):
    X = gen.gaussian_bucket(2, 256, 1024, seed=9) * np.float32(scale)
    out = run_gpu(gns, X)
    for g in range(2):
        assert_parity(out[g], O.orthogonalize(X[g].astype(np.float64)))


@pytest.mark.parametrize("kind", ["low_rank", "student_t", "near_orthogonal", "scaled_1e-3", "scaled_1e+3"])
def test_conditioning_classes(gns, kind):
    """The MoE bucket's classes at its shape (512 x 2048) and seed. An exactly
    rank-32 input sits near the fp16 floor (its null space only holds
    amplified rounding noise); at this shape the error is about 2.9e-2."""
    X = np.stack([gen.moe_matrix(kind, 512, 2048, seed=4000, index=i) for i in range(2)])
    out = run_gpu(gns, X)
    for g in range(2):
        assert_parity(out[g], O.orthogonalize(X[g].astype(np.float64)), what=kind)


def test_ill_conditioned_square(gns):
    X = gen.conditioned_square_bucket(2, 256, seed=3000)
    out = run_gpu(gns, X)
    for g in range(2):
        assert_parity(out[g], O.orthogonalize(X[g].astype(np.float64)))


@pytest.mark.parametrize("steps,restart_at", [(5, 1), (5, 0), (3, 2), (8, 3), (1, 2)])
def test_steps_and_restarts(gns, steps, restart_at):
    X = gen.gaussian_bucket(2, 128, 640, seed=steps * 10 + restart_at)
    out = run_gpu(gns, X, steps=steps, restart_at=restart_at)
    for g in range(2):
        ref = O.gram_ns(X[g].astype(np.float64), steps=steps, restart_at=restart_at)
        assert_parity(out[g], ref, what=f"T={steps} p={restart_at}")


def test_per_step_coefficients(gns):
    coeffs = [(15 / 8, -10 / 8, 3 / 8)] * 4 + [(3.4445, -4.7750, 2.0315)] * 4
    X = gen.gaussian_bucket(2, 96, 384, seed=77)
    out = run_gpu(gns, X, steps=8, restart_at=4, coeffs=coeffs)
    for g in range(2):
        ref = O.gram_ns(X[g].astype(np.float64), steps=8, coeffs=np.array(coeffs).reshape(-1), restart_at=4)
        assert_parity(out[g], ref)


def test_host_buffer_entry_point(gns):
    X = gen.gaussian_bucket(3, 128, 512, seed=12)
    host = torch.from_numpy(X.copy()).pin_memory()
    gns.gns_orthogonalize_batched_host(host)
    dev = run_gpu(gns, X)
    assert np.array_equal(host.numpy(), dev)


def test_nonfinite_input_sets_status(gns):
    X = gen.gaussian_bucket(1, 64, 256, seed=1)
    X[0, 3, 5] = np.inf
    t = torch.from_numpy(X).cuda()
    gns.gns_orthogonalize_batched(t)
    assert gns.gns_get_status() == -3
    assert gns.gns_get_status() == 0  # cleared by the read


def test_invalid_arguments_raise(gns):
    t = torch.zeros(2, 8, 8, device="cuda")
    with pytest.raises(gns.GnsError):
        gns.gns_orthogonalize_batched(t, steps=0)
    with pytest.raises(ValueError):
        gns.gns_orthogonalize_batched(t, steps=2, coeffs=[1.0, 2.0])


def test_restart_schedule_entry_point(gns):
    """Any restart schedule (Dion3 App. B.2.1): the periodic one equals the
    default entry point bit for bit; others match the oracle run with the
    same restart steps; mask bits outside 1 .. steps - 1 are rejected."""
    X = gen.gaussian_bucket(3, 256, 1024, seed=13)
    ref = run_gpu(gns, X)
    t = torch.from_numpy(X.copy()).cuda()
    gns.gns_orthogonalize_batched_schedule(t, 5, (2,))
    torch.cuda.synchronize()
    assert np.array_equal(t.cpu().numpy(), ref)
    for restarts in [(3,), (1,), (2, 3), ()]:
        t = torch.from_numpy(X.copy()).cuda()
        gns.gns_orthogonalize_batched_schedule(t, 5, restarts)
        torch.cuda.synchronize()
        assert gns.gns_get_status() == 0
        out = t.cpu().numpy()
        for g in range(3):
            assert_parity(out[g], O.gram_ns(X[g].astype(np.float64), 5, None, list(restarts)), what=str(restarts))
    with pytest.raises(Exception):
        gns.gns_orthogonalize_batched_schedule(torch.from_numpy(X.copy()).cuda(), 5, (5,))


# Every tile configuration of the GEMM program, forced through GNS_TILE (the
# library picks one by n otherwise): single-CTA 128 x 128 and 128 x 256 tiles
# and CTA pairs. Ragged rectangular and square buckets, so the clipped stores,
# the fp32 output with an addend (last standard-NS step) and the lower-only
# reads all run in each configuration.
TILE_CONFIGS = ["128x1", "256x1", "256x2"]


@pytest.mark.parametrize("tile", TILE_CONFIGS)
@pytest.mark.parametrize("G,R,C", [(2, 520, 1100), (2, 1100, 520), (2, 384, 384)])
def test_forced_tile_configs_match_oracle(gns, monkeypatch, tile, G, R, C):
    monkeypatch.setenv("GNS_TILE", tile)
    X = gen.gaussian_bucket(G, R, C, seed=700 + R + C)
    out = run_gpu(gns, X)
    for g in range(G):
        ref = O.orthogonalize(X[g].astype(np.float64))
        assert_parity(out[g], ref, what=f"{tile} {R}x{C}[{g}]")


def test_result_independent_of_tile_config(gns, monkeypatch):
    """Every tile configuration computes each element with the same k-block
    order and the same epilogue arithmetic, so the results are bitwise equal;
    the library may therefore pick the configuration by bucket size (a matrix
    alone and inside a large bucket can run different configurations) and
    grouped == single still holds bitwise."""
    for G, R, C in ((3, 520, 1100), (2, 1024, 2048), (2, 384, 384)):
        X = gen.gaussian_bucket(G, R, C, seed=900 + R)
        outs = {}
        for tile in TILE_CONFIGS:
            monkeypatch.setenv("GNS_TILE", tile)
            outs[tile] = run_gpu(gns, X)
        ref = outs["256x2"]
        for key, out in outs.items():
            assert np.array_equal(out, ref), (G, R, C, key)
    # Grouped (CTA-pair tiles) against single (128 x 128 tiles, chosen for a
    # lone matrix) with the library's own choice.
    monkeypatch.delenv("GNS_TILE", raising=False)
    X = gen.gaussian_bucket(24, 1024, 2048, seed=901)
    grouped = run_gpu(gns, X)
    for g in (0, 23):
        assert np.array_equal(run_gpu(gns, X[g:g + 1])[0], grouped[g]), g
