"""AdamW kernel vs the fp64 oracle, three consecutive steps with changing
hyper-parameters, parameters in bf16 or fp32 and moments in fp32 or bf16,
tensors of odd sizes and alignments in one launch.  Bars: the updated
parameters within 1e-5 (fp32) or 1e-3 (bf16) of the update's size plus the
oracle's own storage rounding; moments within two storage ulps of their terms."""
import numpy as np
import pytest

from oracle import adamw_oracle as ad
from oracle import muon_oracle as orc
from tests.gpu_util import to_device, to_f64
from workloads import gen_matrix, zeros_matrix

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def mg():
    import __graft_entry__
    __graft_entry__.build()
    import newton_schulz_frobenius_gb300 as pkg
    return pkg


SIZES = [(1, 4096), (1, 7), (64, 200), (3, 33), (1, 1), (1, 30000)]
SCHED = [(1e-3, 0.9, 0.999, 1e-8, 0.01), (5e-4, 0.9, 0.99, 1e-6, 0.0), (2e-3, 0.8, 0.999, 1e-8, 0.1)]


def _store(x64, dtype):
    return x64.astype(np.float32) if dtype == "f32" else orc.bf16_bits_from_f64(orc.round_bf16(x64))


@pytest.mark.parametrize("pdt,sdt", [("f32", "f32"), ("bf16", "f32"), ("bf16", "bf16")])
def test_adamw_matches_oracle(mg, pdt, sdt):
    P = [gen_matrix(700 + i, 1, r, c, 0.5, pdt) for i, (r, c) in enumerate(SIZES)]
    p = [to_device(h, torch).reshape(-1) for h in P]
    m = [to_device(zeros_matrix(r, c, sdt), torch).reshape(-1) for (r, c) in SIZES]
    v = [to_device(zeros_matrix(r, c, sdt), torch).reshape(-1) for (r, c) in SIZES]
    tol = 1e-5 if pdt == "f32" else 1e-3
    for t, (lr, b1, b2, eps, wd) in enumerate(SCHED, start=1):
        G = [gen_matrix(800 + 10 * t + i, 0, r, c, 0.1, pdt) for i, (r, c) in enumerate(SIZES)]
        g = [to_device(h, torch).reshape(-1) for h in G]
        before = [(to_f64(a), to_f64(b), to_f64(c)) for a, b, c in zip(p, m, v)]
        mg.muon_adamw_step(p, g, m, v, lr=lr, beta1=b1, beta2=b2, eps=eps, wd=wd, step=t)
        assert mg.muon_sync_status() == mg.MUON_OK
        F = lambda x: float(np.float32(x))   # noqa: E731  hyper-parameters as the library receives them
        for i in range(len(SIZES)):
            p0, m0, v0 = before[i]
            ref = ad.adamw_step(_store(p0, pdt), G[i].data.reshape(-1), _store(m0, sdt), _store(v0, sdt),
                                lr=F(lr), beta1=F(b1), beta2=F(b2), eps=F(eps), wd=F(wd), step=t,
                                param_dtype=pdt, state_dtype=sdt)
            d = np.linalg.norm(ref["p_exact"] - ref["p_old"])
            err = np.linalg.norm(to_f64(p[i]) - ref["p_exact"]) / d
            q = np.linalg.norm(ref["p_new"] - ref["p_exact"]) / d
            assert err <= tol + q, (i, t, err, q)
            # moments: within two storage ulps of the terms' magnitude (m' = b1 m +
            # (1 - b1) g may cancel, so ulps of the result itself are too strict)
            bits = 8 if sdt == "bf16" else 24
            g64 = orc.to_f64(G[i].data.reshape(-1), pdt)
            for got, want, scale in ((to_f64(m[i]), ref["m_new"], np.abs(F(b1) * m0) + np.abs((1 - F(b1)) * g64)),
                                     (to_f64(v[i]), ref["v_new"], np.abs(F(b2) * v0) + (1 - F(b2)) * g64 * g64)):
                ulp = np.ldexp(1.0, np.floor(np.log2(np.maximum(scale, 1e-30))).astype(int) - (bits - 1))
                assert np.all(np.abs(got - want) <= 2 * ulp + 1e-30), (i, t)


def test_adamw_validation(mg):
    x = torch.zeros(8, device="cuda")
    with pytest.raises(mg.MuonError):
        mg.muon_adamw_step([x], [x], [x], [x], lr=1e-3, step=0)
    with pytest.raises(mg.MuonError):
        mg.muon_adamw_step([x], [x], [x], [x], lr=1e-3, beta1=1.0)
    mg.muon_adamw_step([], [], [], [], lr=1e-3)
