"""The Dion3 update rule on the GPU (Dion3 §6, Algorithm 4, Muon flavor),
through the C ABI, against the oracle: the momentum with its error feedback
bit for bit (which also pins the selected set), the update within the parity
bar, grouped == single, and the f = 1 case against muon_step."""
import numpy as np
import pytest

from gpu_helpers import sr_update_error
from inputs import generators as gen
from oracle import dion3 as D3
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


def bf16_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _inputs(shapes, seed):
    out = []
    for i, (r, c) in enumerate(shapes):
        w, g = gen.muon_param_inputs(r, c, seed=seed, index=i)
        m = gen.gaussian(r, c, seed=seed + 1, index=i, scale=1e-3)
        out.append((torch.from_numpy(w).to(torch.bfloat16), torch.from_numpy(g).to(torch.bfloat16),
                    torch.from_numpy(m)))
    return out


def _run(gns, inputs, fraction, bases, idx_groups=None, seed=3, step=7):
    W = [w.cuda() for w, _, _ in inputs]
    Gr = [g.cuda() for _, g, _ in inputs]
    M = [m.cuda() for _, _, m in inputs]
    for idx in idx_groups or [list(range(len(inputs)))]:
        gns.dion3_step([W[i] for i in idx], [Gr[i] for i in idx], [M[i] for i in idx], fraction, lr=0.02, wd=0.01,
                       mu=0.9, seed=seed, step=step, base_indices=[bases[i] for i in idx])
    torch.cuda.synchronize()
    assert gns.gns_get_status() == 0
    return [bf16_bits(w) for w in W], [m.cpu().numpy() for m in M]


@pytest.mark.parametrize("fraction", [0.25, 0.125, 1.0])
def test_dion3_matches_oracle(gns, fraction):
    shapes = [(256, 1024), (1024, 256), (200, 712), (128, 512), (256, 1024)]  # rows, columns, ragged
    inputs = _inputs(shapes, 61)
    bases = [0, 1 << 33, 1001, 12345, 262144]
    w_gpu, m_gpu = _run(gns, inputs, fraction, bases)
    for i, (r, c) in enumerate(shapes):
        w_bits, g_bits = bf16_bits(inputs[i][0]), bf16_bits(inputs[i][1])
        new_w, new_m, S, O = D3.dion3_step(w_bits, g_bits, inputs[i][2].numpy(), fraction, 0.02, 0.01, 0.9, 3, 7,
                                           bases[i])
        # The momentum (accumulation, then damping of exactly the selected
        # rows or columns) bit for bit: the GPU selected the same set.
        assert np.array_equal(m_gpu[i], new_m), (i, "momentum / selection")
        # The update direction: O on the selected rows (or columns), zero
        # elsewhere; within the parity bar once the rounding noise is out.
        cols = r > c
        full = np.zeros((c, r) if cols else (r, c))
        full[S] = O
        if cols:
            full = full.T
        ok, est, det = sr_update_error(w_gpu[i], w_bits, full, 0.02, 0.01, MU.update_scale(r, c))
        assert ok, (i, est, det)


def test_dion3_grouped_equals_single_bitwise(gns):
    shapes = [(192, 640)] * 3
    inputs = _inputs(shapes, 71)
    bases = [i * 192 * 640 for i in range(3)]
    w_all, m_all = _run(gns, inputs, 0.25, bases)
    w_one, m_one = _run(gns, inputs, 0.25, bases, idx_groups=[[0], [1], [2]])
    for i in range(3):
        assert np.array_equal(w_all[i], w_one[i]) and np.array_equal(m_all[i], m_one[i]), i


def test_dion3_full_fraction_matches_muon(gns):
    """f = 1 selects everything; from zero momentum both optimizers
    orthogonalize G, so the updates agree within the parity bar (the
    selection permutes the rows, which changes rounding only)."""
    shapes = [(256, 1024), (512, 128)]
    inputs = _inputs(shapes, 81)
    inputs = [(w, g, torch.zeros_like(m)) for w, g, m in inputs]
    bases = [0, 256 * 1024]
    w_d3, _ = _run(gns, inputs, 1.0, bases)
    W = [w.cuda() for w, _, _ in inputs]
    gns.muon_step(W, [g.cuda() for _, g, _ in inputs], [m.cuda() for _, _, m in inputs], lr=0.02, wd=0.01, mu=0.9,
                  seed=3, step=7, base_indices=bases)
    torch.cuda.synchronize()
    for i, (r, c) in enumerate(shapes):
        # Both against the orthogonalized gradient: O of the permuted rows is
        # the permuted O, so the f = 1 selection changes rounding only.
        w_bits = bf16_bits(inputs[i][0])
        o_ref = O.orthogonalize(MU.bf16_bits_to_f32(bf16_bits(inputs[i][1])).astype(np.float64))
        for name, got in (("dion3", w_d3[i]), ("muon", bf16_bits(W[i]))):
            ok, est, det = sr_update_error(got, w_bits, o_ref, 0.02, 0.01, MU.update_scale(r, c))
            assert ok, (i, name, est, det)


def test_dion3_rejects_bad_fraction(gns):
    w = torch.zeros(8, 16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(Exception):
        gns.dion3_step([w], [w.clone()], [torch.zeros(8, 16, device="cuda")], 0.0, 0.02, 0.0, 0.9)
