"""Muon elementwise passes and the full Muon step on the GPU, through the C
ABI, against the CPU oracle (bitwise where the arithmetic is fixed)."""
import numpy as np
import pytest

from gpu_helpers import assert_parity, sr_update_error
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


def bf16_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def test_momentum_bitwise(gns):
    for numel in (1, 7, 4096, 100003):
        rng = np.random.default_rng(numel)
        M = rng.standard_normal(numel).astype(np.float32)
        Gv = (1e-3 * rng.standard_normal(numel)).astype(np.float32)
        Gb = torch.from_numpy(Gv).to(torch.bfloat16)
        tM = torch.from_numpy(M).cuda()
        gns.gns_muon_momentum(tM, Gb.cuda(), 0.95)
        want = MU.momentum(M, Gb.float().numpy(), 0.95)
        assert np.array_equal(tM.cpu().numpy(), want)


@pytest.mark.parametrize("rows,cols,base", [(64, 256, 0), (33, 45, 0), (128, 128, 6), (7, 9, 1001), (256, 1024, 1 << 33)])
def test_update_bitwise(gns, rows, cols, base):
    rng = np.random.default_rng(rows * cols + base)
    w = (0.02 * rng.standard_normal((rows, cols))).astype(np.float32)
    o = (rng.standard_normal((rows, cols)) / np.sqrt(cols)).astype(np.float16)
    W = torch.from_numpy(w).to(torch.bfloat16)
    w_bits = bf16_bits(W)
    tW = W.cuda()
    lr, wd, scale, seed, step = 0.02, 0.01, float(MU.update_scale(rows, cols)), 1234567890123, 17
    gns.gns_muon_update(tW, torch.from_numpy(o).cuda(), lr, wd, scale, seed, step, base)
    want = MU.muon_update_bf16(w_bits, o.astype(np.float32), lr, wd, np.float32(scale), seed, step, base)
    assert np.array_equal(bf16_bits(tW), want)


def test_update_shards_match_whole(gns):
    rows, cols = 64, 512
    rng = np.random.default_rng(3)
    W = torch.from_numpy((0.02 * rng.standard_normal((rows, cols))).astype(np.float32)).to(torch.bfloat16).cuda()
    O16 = torch.from_numpy((rng.standard_normal((rows, cols)) / 20).astype(np.float16)).cuda()
    whole = W.clone()
    gns.gns_muon_update(whole, O16, 0.02, 0.01, 2.0, 5, 6, 1000)
    top, bot = W[:24].clone(), W[24:].clone()
    gns.gns_muon_update(top, O16[:24].contiguous(), 0.02, 0.01, 2.0, 5, 6, 1000)
    gns.gns_muon_update(bot, O16[24:].contiguous(), 0.02, 0.01, 2.0, 5, 6, 1000 + 24 * cols)
    assert torch.equal(torch.cat([top, bot]), whole)


@pytest.mark.parametrize("p", [0.1, 0.25, 0.5])
def test_sr_unbiased_on_gpu(gns, p):
    """Muon kernel card: a sub-ULP update over 2e5 bf16 elements averages to
    the true value. W = 1 + p ULP is built as (1 - lr wd) W - lr s O with
    W = 1, wd = 0, lr s O = -p ULP exactly."""
    n = 200_000
    ulp = 2.0 ** -7
    errs = []
    for k in range(16):
        W = torch.ones(1, n, dtype=torch.bfloat16, device="cuda")
        # o = -p * ulp / (lr * scale) with lr = 1, scale = 2^-10: fp16-exact for p in {0.1 (rounded), 0.25, 0.5}
        o = torch.full((1, n), -p * ulp * 1024.0, dtype=torch.float16, device="cuda")
        # The fp32 value the kernel rounds: 1 - fl(2^-10 * o), each step exact or rounded once.
        target = float(np.float32(1.0) - np.float32(2.0 ** -10) * np.float32(o[0, 0].item()))
        gns.gns_muon_update(W, o, 1.0, 0.0, 2.0 ** -10, 100 + k, k, 0)
        errs.append((W.float().double().mean().item() - target) / ulp)
    assert abs(np.mean(errs)) < 1e-3


def test_muon_step_matches_oracle(gns):
    shapes = [(128, 512), (512, 128), (128, 512), (256, 256), (96, 200)]
    rng_seed = 21
    Ws, Gs, Ms = [], [], []
    for i, (r, c) in enumerate(shapes):
        w, g = gen.muon_param_inputs(r, c, seed=rng_seed, index=i)
        Ws.append(torch.from_numpy(w).to(torch.bfloat16))
        Gs.append(torch.from_numpy(g).to(torch.bfloat16))
        Ms.append(torch.from_numpy(np.random.default_rng(i).standard_normal((r, c)).astype(np.float32) * 1e-3))
    w_bits = [bf16_bits(w) for w in Ws]
    g_bits = [bf16_bits(g) for g in Gs]
    m_np = [m.numpy().copy() for m in Ms]
    dW = [w.cuda() for w in Ws]
    dG = [g.cuda() for g in Gs]
    dM = [m.cuda() for m in Ms]
    bases = [1000 * i for i in range(len(shapes))]
    gns.muon_step(dW, dG, dM, lr=0.02, wd=0.01, mu=0.95, seed=0, step=3, base_indices=bases)
    torch.cuda.synchronize()
    assert gns.gns_get_status() == 0
    new_w, new_m, outs = MU.muon_step(w_bits, g_bits, m_np, 0.02, 0.01, 0.95, 0, 3, bases)
    for i, (r, c) in enumerate(shapes):
        assert np.array_equal(dM[i].cpu().numpy(), new_m[i]), f"momentum {i}"
        # The update direction is the orthogonalized momentum: the update
        # within the parity bar once the rounding noise is taken out.
        ok, est, det = sr_update_error(bf16_bits(dW[i]), w_bits[i], outs[i], 0.02, 0.01, MU.update_scale(r, c))
        assert ok, (i, est, det)


def test_fused_update_matches_separate_pass_bitwise(gns, monkeypatch):
    """The Muon update fused into the last product's epilogue gives the same
    bits as the separate pass over a stored fp16 O (same rounding of O, same
    Philox counters), for aligned and unaligned global index bases, ragged,
    transposed and square matrices."""
    shapes = [(128, 512), (512, 128), (96, 200), (256, 256), (130, 4100), (200, 200)]
    bases = [0, 1 << 33, 1001, 4 * 10 ** 6 + 2, 7, 123456789]
    inputs = []
    for i, (r, c) in enumerate(shapes):
        w, g = gen.muon_param_inputs(r, c, seed=31, index=i)
        m = gen.gaussian(r, c, seed=32, index=i, scale=1e-3)
        inputs.append((torch.from_numpy(w).to(torch.bfloat16), torch.from_numpy(g).to(torch.bfloat16),
                       torch.from_numpy(m)))

    def run(fused):
        monkeypatch.setenv("GNS_MUON_FUSED", "1" if fused else "0")
        W = [w.cuda() for w, _, _ in inputs]
        Gr = [g.cuda() for _, g, _ in inputs]
        M = [m.cuda() for _, _, m in inputs]
        gns.muon_step(W, Gr, M, lr=0.02, wd=0.01, mu=0.95, seed=5, step=11, base_indices=bases)
        torch.cuda.synchronize()
        assert gns.gns_get_status() == 0
        return [bf16_bits(w) for w in W], [m.cpu().numpy() for m in M]

    w_sep, m_sep = run(False)
    w_fused, m_fused = run(True)
    for i in range(len(shapes)):
        assert np.array_equal(m_sep[i], m_fused[i]), shapes[i]
        assert np.array_equal(w_sep[i], w_fused[i]), shapes[i]


def _normuon_inputs(shapes, seed):
    out = []
    for i, (r, c) in enumerate(shapes):
        w, g = gen.muon_param_inputs(r, c, seed=seed, index=i)
        m = gen.gaussian(r, c, seed=seed + 1, index=i, scale=1e-3)
        v = np.abs(gen.gaussian(r, 1, seed=seed + 2, index=i, scale=1e-4))[:, 0]  # a previous step's state
        out.append((torch.from_numpy(w).to(torch.bfloat16), torch.from_numpy(g).to(torch.bfloat16),
                    torch.from_numpy(m), torch.from_numpy(v.astype(np.float32))))
    return out


def test_normuon_step_matches_oracle(gns):
    """NorMuon (Dion3 Eq. 2) against the oracle: momentum bitwise; the row
    second moments and the update within the parity bar (they follow O)."""
    shapes = [(128, 512), (512, 128), (96, 200), (256, 256), (128, 512)]
    inputs = _normuon_inputs(shapes, 41)
    bases = [0, 1 << 33, 1001, 5, 70000]
    W = [w.cuda() for w, _, _, _ in inputs]
    Gr = [g.cuda() for _, g, _, _ in inputs]
    M = [m.cuda() for _, _, m, _ in inputs]
    V = [v.cuda() for _, _, _, v in inputs]
    gns.normuon_step(W, Gr, M, V, lr=0.02, wd=0.01, mu=0.95, beta2=0.95, eps=1e-8, seed=0, step=3,
                     base_indices=bases)
    torch.cuda.synchronize()
    assert gns.gns_get_status() == 0
    w_bits = [bf16_bits(w) for w, _, _, _ in inputs]
    new_w, new_m, new_v, dirs = MU.normuon_step(w_bits, [bf16_bits(g) for _, g, _, _ in inputs],
                                                [m.numpy() for _, _, m, _ in inputs],
                                                [v.numpy().astype(np.float64) for _, _, _, v in inputs],
                                                0.02, 0.01, 0.95, 0.95, 1e-8, 0, 3, bases)
    for i, (r, c) in enumerate(shapes):
        assert np.array_equal(M[i].cpu().numpy(), new_m[i]), f"momentum {i}"
        v_got = V[i].cpu().numpy().astype(np.float64)
        assert np.linalg.norm(v_got - new_v[i]) <= 6e-2 * np.linalg.norm(new_v[i]), (i, "second moment")
        ok, est, det = sr_update_error(bf16_bits(W[i]), w_bits[i], dirs[i], 0.02, 0.01, MU.update_scale(r, c))
        assert ok, (i, est, det)


def test_normuon_grouped_equals_single_bitwise(gns):
    shapes = [(192, 320)] * 3
    inputs = _normuon_inputs(shapes, 51)

    def run(groups):
        W = [w.cuda() for w, _, _, _ in inputs]
        Gr = [g.cuda() for _, g, _, _ in inputs]
        M = [m.cuda() for _, _, m, _ in inputs]
        V = [v.cuda() for _, _, _, v in inputs]
        bases = [i * 192 * 320 for i in range(3)]
        for idx in groups:
            gns.normuon_step([W[i] for i in idx], [Gr[i] for i in idx], [M[i] for i in idx], [V[i] for i in idx],
                             lr=0.02, wd=0.01, mu=0.95, seed=9, step=4, base_indices=[bases[i] for i in idx])
        torch.cuda.synchronize()
        assert gns.gns_get_status() == 0
        return [bf16_bits(w) for w in W], [v.cpu().numpy() for v in V]

    w_all, v_all = run([[0, 1, 2]])
    w_one, v_one = run([[0], [1], [2]])
    for i in range(3):
        assert np.array_equal(w_all[i], w_one[i]) and np.array_equal(v_all[i], v_one[i]), i
