"""The GEMM program's tile claiming does not depend on how many of its CTAs are
resident: a tile waits only for tiles with smaller tickets, which running CTAs
have already claimed. Here another stream keeps the GPU busy with a long
matrix-multiply loop while a bucket runs, so the program starts with only
part of the machine; the call must end with status 0, match the oracle and
give the same bits as the same call on a quiet GPU (every tile's reduction
order is fixed, whichever CTA computes it)."""
import numpy as np
import pytest

from gpu_helpers import assert_parity
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


def busy_loop(stream, n, iters):
    """Queue `iters` bf16 matrix products of n x n on `stream`."""
    with torch.cuda.stream(stream):
        a = torch.randn(n, n, device="cuda", dtype=torch.bfloat16)
        b = torch.randn(n, n, device="cuda", dtype=torch.bfloat16)
        for _ in range(iters):
            a = torch.matmul(a, b) * (n ** -0.5)
    return a


@pytest.mark.parametrize("shape", [(8, 1024, 4096), (12, 2048, 2048), (6, 1021, 4093)],
                         ids=["8x1024x4096", "12x2048x2048", "6x1021x4093"])
def test_bucket_alongside_a_busy_stream(gns, shape):
    G, R, C = shape
    X = gen.gaussian_bucket(G, R, C, seed=7100 + R)
    x32 = torch.from_numpy(np.ascontiguousarray(X, dtype=np.float32)).cuda()

    quiet = x32.clone()
    gns.gns_orthogonalize_batched(quiet)
    torch.cuda.synchronize()
    assert gns.gns_get_status() == 0

    side = torch.cuda.Stream()
    outs = []
    for rep in range(3):
        # The side stream's work is queued first, so the bucket's kernels
        # start while the products hold most of the SMs.
        busy = busy_loop(side, 8192, 40)
        t = x32.clone()
        gns.gns_orthogonalize_batched(t)
        outs.append(t)
        torch.cuda.synchronize()
        assert gns.gns_get_status() == 0, gns.gns_last_error()
        assert bool(torch.isfinite(busy.float()).all())
    for rep, t in enumerate(outs):
        assert torch.equal(t, quiet), f"repeat {rep} differs from the quiet run"
    out = quiet.cpu().numpy()
    for g in range(G):
        assert_parity(out[g], O.orthogonalize(X[g].astype(np.float64)), what=f"matrix {g}")


CHILD = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
sys.path.insert(0, sys.argv[1] + "/tests")
import test_gpu_residency as T
import newton_schulz_gram_gb300 as gns
gns.load()
np.savez(sys.argv[2], *T.grid_workload(gns))
"""


def grid_workload(gns):
    """Muon and NorMuon steps (separate update pass) and the standalone update
    on shapes whose rows are 1000 columns wide, so that a small grid's stride
    (a multiple of 8 elements) crosses rows at varying columns; returns every
    output as host arrays."""
    import os
    os.environ["GNS_MUON_FUSED"] = "0"
    shapes = [(600, 1000), (600, 1000), (1000, 520)]
    outs = []
    for kind in ("muon", "normuon"):
        W, Gr, M, V = [], [], [], []
        for i, (r, c) in enumerate(shapes):
            w, g = gen.muon_param_inputs(r, c, seed=81, index=i)
            W.append(torch.from_numpy(w).to(torch.bfloat16).cuda())
            Gr.append(torch.from_numpy(g).to(torch.bfloat16).cuda())
            M.append(torch.from_numpy(gen.gaussian(r, c, seed=82, index=i, scale=1e-3)).cuda())
            V.append(torch.full((r,), 1e-8, device="cuda"))
        bases = [0, 600 * 1000 + 8, 1 << 33]
        if kind == "muon":
            gns.muon_step(W, Gr, M, lr=0.02, wd=0.01, mu=0.95, seed=3, step=5, base_indices=bases)
        else:
            gns.normuon_step(W, Gr, M, V, lr=0.02, wd=0.01, mu=0.95, seed=3, step=5, base_indices=bases)
        torch.cuda.synchronize()
        assert gns.gns_get_status() == 0
        outs += [w.view(torch.int16).cpu().numpy() for w in W] + [v.cpu().numpy() for v in V]
    w = (0.02 * torch.randn(3000, 1000, generator=torch.Generator().manual_seed(4))).to(torch.bfloat16).cuda()
    o = torch.randn(3000, 1000, generator=torch.Generator().manual_seed(5)).to(torch.float16).cuda()
    gns.gns_muon_update(w, o, 0.02, 0.01, 0.5, 7, 9, 1 << 20)
    torch.cuda.synchronize()
    assert gns.gns_get_status() == 0
    outs.append(w.view(torch.int16).cpu().numpy())
    os.environ.pop("GNS_MUON_FUSED")
    return outs


def test_results_independent_of_grid_size(gns, tmp_path):
    """The same Muon, NorMuon and update calls on the whole GPU and in a child
    process whose launches are capped at two SMs (each thread of the update
    pass then strides through many rows; the GEMM program runs on one CTA
    pair): bitwise equal outputs."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    full = grid_workload(gns)
    out = tmp_path / "small_grid.npz"
    env = dict(os.environ, GNS_NUM_SMS="2")
    r = subprocess.run([sys.executable, "-c", CHILD, root, str(out)], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    small = np.load(out)
    assert len(small.files) == len(full)
    for i, a in enumerate(full):
        assert np.array_equal(small[f"arr_{i}"], a), f"output {i} differs between grid sizes"


def test_results_independent_of_claim_pacing(gns, monkeypatch):
    """How far ahead of its producer a pair claims tiles (GNS_LOOKAHEAD)
    changes which pair computes which tile, never a tile's arithmetic: the
    outputs are bitwise equal for lookaheads 1, 3 and 8."""
    X = gen.gaussian_bucket(10, 1024, 2048, seed=7400)
    outs = {}
    for la in ("1", "3", "8"):
        monkeypatch.setenv("GNS_LOOKAHEAD", la)
        t = torch.from_numpy(np.ascontiguousarray(X, dtype=np.float32)).cuda()
        gns.gns_orthogonalize_batched(t)
        torch.cuda.synchronize()
        assert gns.gns_get_status() == 0
        outs[la] = t.cpu().numpy()
    assert np.array_equal(outs["1"], outs["3"]) and np.array_equal(outs["1"], outs["8"])
