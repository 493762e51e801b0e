"""The pages' workloads at their full sizes, each run as one bucket through the
C ABI in the launch configuration the benchmark times, against the fp64
oracle matrix by matrix (Dion3 Algorithm 3 for rectangular matrices,
Algorithm 1 for square ones; Dion3 Eq. 1 and Section 6 for the Muon step).

The rectangular and square buckets are checked whole. The 7B Muon step
(224 matrices, 6.98e9 parameters) is checked on a sample of matrices, one or
more per shape; every other matrix of it is checked for finiteness and
against the properties below, which hold at any size."""
import numpy as np
import pytest

from gpu_helpers import assert_parity, parity_metrics, sr_update_error
from inputs import generators as gen
from oracle import gram_ns as O
from oracle import muon as MU

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gns():
    import newton_schulz_gram_gb300 as m
    from newton_schulz_gram_gb300 import build
    build.build()
    m.load()
    return m


def run_bucket(gns, X):
    t = torch.from_numpy(np.ascontiguousarray(X, dtype=np.float32)).cuda()
    gns.gns_orthogonalize_batched(t)
    torch.cuda.synchronize()
    assert gns.gns_get_status() == 0
    return t


def polar_alignment(O_, X):
    """O = p(X X^T) X for an odd polynomial iteration, so O X^T is symmetric
    and positive semi-definite up to the method's error: returns the relative
    asymmetry ||A - A^T|| / ||A|| and the trace of A = O X^T (>= 0)."""
    A = O_ @ X.T if X.shape[0] <= X.shape[1] else X.T @ O_
    asym = torch.linalg.matrix_norm(A - A.T) / torch.linalg.matrix_norm(A)
    return float(asym), float(torch.trace(A))


@pytest.mark.parametrize("name", ["mlp_24x1024x4096", "square_16x2048"])
def test_whole_bucket_against_oracle(gns, name):
    X = gen.config_bucket(name)
    out = run_bucket(gns, X).cpu().numpy()
    assert np.isfinite(out).all()
    for g in range(X.shape[0]):
        assert_parity(out[g], O.orthogonalize(X[g].astype(np.float64)), what=f"{name}[{g}]")


def test_moe_bucket_against_oracle(gns):
    """256 matrices 512 x 2048 in six input classes (43, 43, 43, 43, 42, 42)."""
    name = "moe_256x512x2048"
    X = gen.config_bucket(name)
    out = run_bucket(gns, X).cpu().numpy()
    assert np.isfinite(out).all()
    worst = {}
    for g in range(X.shape[0]):
        kind = gen.moe_class_of(g, X.shape[0])
        m = parity_metrics(out[g], O.orthogonalize(X[g].astype(np.float64)))
        w = worst.setdefault(kind, dict(rel=0.0, cos=1.0, sv=0.0))
        w["rel"] = max(w["rel"], m["rel"])
        w["cos"] = min(w["cos"], m["cos"])
        w["sv"] = max(w["sv"], m["sv"])
    print({k: {kk: round(vv, 5) for kk, vv in v.items()} for k, v in worst.items()})
    for kind, w in worst.items():
        assert w["rel"] <= 3e-2 and w["cos"] >= 0.98 and w["sv"] <= 0.05, (kind, w)


def bf16_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def test_llama7b_muon_step(gns):
    """One Muon step over the 7B Llama-like stack: 32 layers of q, o (4096^2),
    k, v (1024 x 4096), gate, up (14336 x 4096) and down (4096 x 14336); bf16
    W ~ N(0, 0.02), bf16 G ~ N(0, 1e-3), fp32 M; mu = 0.95, lr = 0.02,
    wd = 0.01. The sampled matrices come from the seeded input generators and
    are checked against the oracle (momentum bitwise; the update within the
    parity bar once the expected stochastic-rounding noise is taken out, see
    sr_update_error); the others are filled from a seeded device generator
    and checked for finiteness."""
    shapes = gen.llama7b_shapes()
    sampled = {"layer0.q", "layer0.k", "layer0.gate", "layer31.down"}
    seed = 5000
    dev_gen = torch.Generator(device="cuda")
    dev_gen.manual_seed(seed)
    W, Gr, M, host = [], [], [], {}
    for i, (name, r, c) in enumerate(shapes):
        if name in sampled:
            w, g = gen.muon_param_inputs(r, c, seed=seed, index=i)
            m = gen.gaussian(r, c, seed=seed + 1, index=i, scale=1e-3)
            wt, gt = torch.from_numpy(w).to(torch.bfloat16), torch.from_numpy(g).to(torch.bfloat16)
            host[i] = (bf16_bits(wt), bf16_bits(gt), m.copy())
            W.append(wt.cuda())
            Gr.append(gt.cuda())
            M.append(torch.from_numpy(m).cuda())
        else:
            W.append((0.02 * torch.randn(r, c, device="cuda", generator=dev_gen)).to(torch.bfloat16))
            Gr.append((1e-3 * torch.randn(r, c, device="cuda", generator=dev_gen)).to(torch.bfloat16))
            M.append(1e-3 * torch.randn(r, c, device="cuda", generator=dev_gen))
    bases, acc = [], 0
    for w in W:
        bases.append(acc)
        acc += w.numel()
    assert acc == 6_979_321_856
    gns.muon_step(W, Gr, M, lr=0.02, wd=0.01, mu=0.95, seed=0, step=2, base_indices=bases)
    torch.cuda.synchronize()
    assert gns.gns_get_status() == 0
    for i in range(len(shapes)):
        assert bool(torch.isfinite(M[i]).all()) and bool(torch.isfinite(W[i].float()).all()), shapes[i][0]
    for i, (w_bits, g_bits, m0) in host.items():
        name, r, c = shapes[i]
        new_w, new_m, outs = MU.muon_step([w_bits], [g_bits], [m0], 0.02, 0.01, 0.95, 0, 2, [bases[i]])
        assert np.array_equal(M[i].cpu().numpy(), new_m[0]), f"momentum {name}"
        ok, est, det = sr_update_error(bf16_bits(W[i]), w_bits, outs[0], 0.02, 0.01, MU.update_scale(r, c))
        assert ok, (name, est, det)


def test_per_head_split_bucket(gns):
    """An attention projection split by head (Dion3 App. A.1.1): W_Q of a
    d = 4096 model with H = 16 heads becomes 16 matrices of 256 x 4096, whose
    aspect ratio alpha = H makes the Gram form cheap. Every matrix against the
    oracle."""
    X = gen.gaussian_bucket(16, 256, 4096, seed=6000)
    out = run_bucket(gns, X).cpu().numpy()
    for g in range(X.shape[0]):
        assert_parity(out[g], O.orthogonalize(X[g].astype(np.float64)), what=f"head {g}")


def llama7b_bucket(kind):
    """The n = 4096 shapes of the 7B stack (Dion3 Fig. 1 workload): two
    square 4096 x 4096 matrices (Gaussian, and a log-uniform [1e-6, 1]
    spectrum with Haar singular vectors), the 4096 x 14336 down projection and
    the 14336 x 4096 gate / up projection (transposed on the way in)."""
    if kind == "square_4096":
        return np.stack([gen.gaussian(4096, 4096, 5100, 0), gen.log_uniform_spectrum(4096, 5100, 1)])
    if kind == "down_4096x14336":
        return gen.gaussian_bucket(1, 4096, 14336, seed=5101)
    return gen.gaussian_bucket(1, 14336, 4096, seed=5102)


@pytest.mark.parametrize("kind", ["square_4096", "down_4096x14336", "gate_14336x4096"])
def test_llama7b_shapes_against_oracle(gns, kind):
    """gns_orthogonalize_batched on the 7B stack's n = 4096 shapes in the
    library's default tile configuration, each matrix against the oracle at
    the parity bar (relative error, cosine, singular values): the direct
    check of the largest shapes, where the fp16 state is prescaled the most."""
    X = llama7b_bucket(kind)
    out = run_bucket(gns, X).cpu().numpy()
    for g in range(X.shape[0]):
        m = assert_parity(out[g], O.orthogonalize(X[g].astype(np.float64)), what=f"{kind}[{g}]")
        print(kind, g, {k: round(v, 5) if isinstance(v, float) else v for k, v in m.items()})
